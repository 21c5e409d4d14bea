// CPU oracle for the MoE layer of a speculative-decoding verify round.
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
// benchmark's CPU-baseline leg may load this file's library.  It shares no code with
// the CUDA path: every conversion and every loop below is written out here.
//
// What it computes (sources: "How AlphaInfer makes local decoding fast", sections 1
// and 3.1 -- a verify round over 1..16 token rows, where each extra row routes to
// experts the other rows did not need; "infero", the decoder-block diagram
// (silu(W_g x) * (W_u x) -> W_d) and "Design notes" (weights consumed in their
// 32-element block encoding, block scales folded in in float)):
//
//   a1  logits[r][e] = sum_h Wr[e][h] * x[r][h] in fp32, in the canonical order below.
//   a2  per row, the k largest logits ordered by (logit desc, id asc); weights
//       w_j = exp(l_j - l_1) / sum_i exp(l_i - l_1) over the k picks.
//   a3  union U = ascending distinct ids over all rows' picks.
//   a4  for each routed (row, expert): g = Wg x, v = Wu x, h = silu(g) * v,
//       silu(g) = g / (1 + exp(-g)), with W = fp16 scale * int4 code.
//   a5  y = Wd h;  out[r] = sum_j w_j * y_{r, ids[r][j]}  (j in rank order).
//   Optional routing tail skip (Avalon README, "Numbers" for the RX 7900 XT: experts
//   that every token of a verification routes only at rank 7 or lower are skipped):
//   with threshold T > 0, a union expert is dropped when every row that picked it has
//   it at 1-based rank >= T; the picks of dropped experts contribute nothing and the
//   remaining weights are not renormalised (the page says nothing about it).
//
// Precision (readings of points the pages leave open; each is listed in the design
// notes):
//   * Router logits are fp32 with a fixed summation order, because the top-k
//     decision must be bit-identical on CPU and GPU: 32 lane partials, lane l takes
//     elements 128c + 4l + j (c ascending, j = 0..3) with a correctly rounded fma each;
//     then partials are combined by the xor-butterfly p_l <- p_l + p_{l^o},
//     o = 16, 8, 4, 2, 1, and the logit is p_0.  H must be a multiple of 128.
//   * Everything after the routing decision (softmax weights, expert FFN, combine)
//     is evaluated in fp64 from the exact fp32 dequantized weights, so the oracle's
//     own rounding is far below the 2e-3 / 1e-3 output tolerance.
//   * Dequantized weight = (float)fp16_scale * (float)q, q in [-8, 7]; exact in fp32.
//
// Build: g++ -O2 -ffp-contract=off (no fast-math), single-threaded.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// IEEE binary16 bits -> double (exact).
double half_bits_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int ex = (b >> 10) & 0x1f;
  int man = b & 0x3ff;
  double v;
  if (ex == 0) {
    v = std::ldexp((double)man, -24);  // subnormal or zero
  } else if (ex == 31) {
    v = man ? NAN : INFINITY;
  } else {
    v = std::ldexp((double)(man + 1024), ex - 25);
  }
  return sign ? -v : v;
}

// bfloat16 bits -> float (exact: the 16 bits are the high half of the fp32 pattern).
float bf16_bits_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// a1: one router logit in the canonical fp32 order.
float canonical_logit(const float* w, const float* x, int H) {
  float p[32];
  for (int l = 0; l < 32; ++l) p[l] = 0.0f;
  for (int c = 0; c < H / 128; ++c)
    for (int l = 0; l < 32; ++l)
      for (int j = 0; j < 4; ++j) {
        int h = 128 * c + 4 * l + j;
        p[l] = std::fma(w[h], x[h], p[l]);
      }
  for (int o = 16; o >= 1; o >>= 1) {
    float q[32];
    for (int l = 0; l < 32; ++l) q[l] = p[l] + p[l ^ o];
    for (int l = 0; l < 32; ++l) p[l] = q[l];
  }
  return p[0];
}

// a2 ordering: true if (la, ia) ranks before (lb, ib).  -0.0 == +0.0 here, so a
// signed-zero pair is a tie and the lower id wins.
bool ranks_before(float la, int ia, float lb, int ib) {
  return la > lb || (la == lb && ia < ib);
}

struct Routing {
  std::vector<float> logits;  // [R][E]
  std::vector<int32_t> ids;   // [R][k]
  std::vector<double> w;      // [R][k]
  std::vector<char> keep;     // [R][k]: the pick's expert is evaluated (not tail-skipped)
  std::vector<int32_t> uni;   // ascending, after the tail skip
  std::vector<double> gap64;  // [R]
};

int route(int H, int E, int k, int R, const float* router, const uint16_t* xb, Routing& out,
          int tail_rank = 0) {
  if (H <= 0 || H % 128 || E <= 0 || k <= 0 || k > E || R <= 0) return -1;
  out.logits.assign((size_t)R * E, 0.0f);
  out.ids.assign((size_t)R * k, -1);
  out.w.assign((size_t)R * k, 0.0);
  out.gap64.assign(R, 0.0);
  std::vector<float> x(H);
  std::vector<char> hit(E, 0);
  for (int r = 0; r < R; ++r) {
    for (int h = 0; h < H; ++h) x[h] = bf16_bits_to_float(xb[(size_t)r * H + h]);
    float* lg = &out.logits[(size_t)r * E];
    for (int e = 0; e < E; ++e) lg[e] = canonical_logit(router + (size_t)e * H, x.data(), H);
    // top-k by repeated selection of the best remaining expert
    std::vector<char> taken(E, 0);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || ranks_before(lg[e], e, lg[best], best))) best = e;
      taken[best] = 1;
      out.ids[(size_t)r * k + j] = best;
      hit[best] = 1;
    }
    // softmax restricted to the k picks, shifted by the largest logit
    const int32_t* id = &out.ids[(size_t)r * k];
    double l1 = (double)lg[id[0]], den = 0.0;
    std::vector<double> ex(k);
    for (int j = 0; j < k; ++j) {
      ex[j] = std::exp((double)lg[id[j]] - l1);
      den += ex[j];
    }
    for (int j = 0; j < k; ++j) out.w[(size_t)r * k + j] = ex[j] / den;
    // fp64 shadow: exact-order logits, gap between k-th and (k+1)-th
    if (k < E) {
      std::vector<double> l64(E);
      for (int e = 0; e < E; ++e) {
        double s = 0.0;
        for (int h = 0; h < H; ++h) s += (double)router[(size_t)e * H + h] * (double)x[h];
        l64[e] = s;
      }
      std::vector<char> t2(E, 0);
      double kth = 0.0, next = 0.0;
      for (int j = 0; j <= k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e)
          if (!t2[e] && (best < 0 || l64[e] > l64[best])) best = e;
        t2[best] = 1;
        if (j == k - 1) kth = l64[best];
        if (j == k) next = l64[best];
      }
      out.gap64[r] = kth - next;
    } else {
      out.gap64[r] = INFINITY;
    }
  }
  // tail skip: an expert survives if some row picked it at 1-based rank < tail_rank
  std::vector<char> alive(E, 0);
  for (int r = 0; r < R; ++r)
    for (int j = 0; j < k; ++j)
      if (tail_rank <= 0 || j + 1 < tail_rank) alive[out.ids[(size_t)r * k + j]] = 1;
  out.keep.assign((size_t)R * k, 0);
  for (int r = 0; r < R; ++r)
    for (int j = 0; j < k; ++j) out.keep[(size_t)r * k + j] = alive[out.ids[(size_t)r * k + j]];
  out.uni.clear();
  for (int e = 0; e < E; ++e)
    if (hit[e] && alive[e]) out.uni.push_back(e);
  return 0;
}

// a4 + a5 for one (row, expert): y[H] = Wd (silu(Wg x) * (Wu x)), in fp64.
void expert_ffn(int H, int I, const float* x, const int8_t* qg, const uint16_t* sg,
                const int8_t* qu, const uint16_t* su, const int8_t* qd, const uint16_t* sd,
                double* y) {
  std::vector<double> hv(I);
  for (int i = 0; i < I; ++i) {
    double g = 0.0, v = 0.0;
    for (int b = 0; b < H / 32; ++b) {
      float sgb = (float)half_bits_to_double(sg[(size_t)i * (H / 32) + b]);
      float sub = (float)half_bits_to_double(su[(size_t)i * (H / 32) + b]);
      for (int t = 0; t < 32; ++t) {
        int h = 32 * b + t;
        float wg = sgb * (float)qg[(size_t)i * H + h];
        float wu = sub * (float)qu[(size_t)i * H + h];
        g += (double)wg * (double)x[h];
        v += (double)wu * (double)x[h];
      }
    }
    hv[i] = g / (1.0 + std::exp(-g)) * v;
  }
  for (int o = 0; o < H; ++o) {
    double acc = 0.0;
    for (int b = 0; b < I / 32; ++b) {
      float sdb = (float)half_bits_to_double(sd[(size_t)o * (I / 32) + b]);
      for (int t = 0; t < 32; ++t) {
        int i = 32 * b + t;
        float wd = sdb * (float)qd[(size_t)o * I + i];
        acc += (double)wd * hv[i];
      }
    }
    y[o] = acc;
  }
}

struct Provided {
  int P;
  const int32_t* ids;
  const int8_t *qg, *qu, *qd;
  const uint16_t *sg, *su, *sd;
  int index_of(int e) const {
    for (int p = 0; p < P; ++p)
      if (ids[p] == e) return p;
    return -1;
  }
};

void ffn_of(int H, int I, const Provided& pv, int p, const float* x, double* y) {
  size_t nq = (size_t)H * I, ns = nq / 32;
  expert_ffn(H, I, x, pv.qg + p * nq, pv.sg + p * ns, pv.qu + p * nq, pv.su + p * ns,
             pv.qd + p * nq, pv.sd + p * ns, y);
}

}  // namespace

extern "C" {

int oracle_route_tail(int H, int E, int k, int R, int tail_rank, const float* router,
                      const uint16_t* x_bf16, float* logits, int32_t* ids, double* w, uint8_t* keep,
                      int32_t* union_ids, int32_t* n_union, double* gap64);
int oracle_layer_tail(int H, int E, int k, int I, int R, int tail_rank, const float* router,
                      const uint16_t* x_bf16, int P, const int32_t* prov_ids, const int8_t* qg,
                      const uint16_t* sg, const int8_t* qu, const uint16_t* su, const int8_t* qd,
                      const uint16_t* sd, double* out);
int oracle_layer_dense_tail(int H, int E, int k, int I, int R, int tail_rank, const float* router,
                            const uint16_t* x_bf16, const int8_t* qg, const uint16_t* sg,
                            const int8_t* qu, const uint16_t* su, const int8_t* qd,
                            const uint16_t* sd, double* out);

double oracle_half_to_double(uint16_t b) { return half_bits_to_double(b); }
float oracle_bf16_to_float(uint16_t b) { return bf16_bits_to_float(b); }

float oracle_canonical_logit(const float* w, const float* x, int H) {
  if (H <= 0 || H % 128) return NAN;
  return canonical_logit(w, x, H);
}

// a1-a3.  Outputs: logits [R][E] fp32, ids [R][k], w [R][k] fp64, union [E] (first
// *n_union entries valid), gap64 [R] (may be NULL).  Returns 0, or -1 on bad dims.
int oracle_route(int H, int E, int k, int R, const float* router, const uint16_t* x_bf16,
                 float* logits, int32_t* ids, double* w, int32_t* union_ids, int32_t* n_union,
                 double* gap64) {
  return oracle_route_tail(H, E, k, R, 0, router, x_bf16, logits, ids, w, nullptr, union_ids,
                           n_union, gap64);
}

// oracle_route with the tail skip at threshold tail_rank (0 = off); keep [R][k] (may be
// NULL) receives 1 for picks whose expert is evaluated.
int oracle_route_tail(int H, int E, int k, int R, int tail_rank, const float* router,
                      const uint16_t* x_bf16, float* logits, int32_t* ids, double* w, uint8_t* keep,
                      int32_t* union_ids, int32_t* n_union, double* gap64) {
  Routing rt;
  if (route(H, E, k, R, router, x_bf16, rt, tail_rank)) return -1;
  if (keep)
    for (size_t i = 0; i < rt.keep.size(); ++i) keep[i] = (uint8_t)rt.keep[i];
  std::memcpy(logits, rt.logits.data(), rt.logits.size() * sizeof(float));
  std::memcpy(ids, rt.ids.data(), rt.ids.size() * sizeof(int32_t));
  std::memcpy(w, rt.w.data(), rt.w.size() * sizeof(double));
  for (size_t i = 0; i < rt.uni.size(); ++i) union_ids[i] = rt.uni[i];
  *n_union = (int32_t)rt.uni.size();
  if (gap64) std::memcpy(gap64, rt.gap64.data(), rt.gap64.size() * sizeof(double));
  return 0;
}

// a1-a5 over the union.  The caller provides the weights of P experts (ids
// prov_ids[P]; qg/qu [P][I][H], sg/su [P][I][H/32], qd [P][H][I], sd [P][H][I/32]).
// Returns 0, -1 on bad dims, -2 if a routed expert is not among the provided ones.
int oracle_layer(int H, int E, int k, int I, int R, const float* router, const uint16_t* x_bf16,
                 int P, const int32_t* prov_ids, const int8_t* qg, const uint16_t* sg,
                 const int8_t* qu, const uint16_t* su, const int8_t* qd, const uint16_t* sd,
                 double* out) {
  return oracle_layer_tail(H, E, k, I, R, 0, router, x_bf16, P, prov_ids, qg, sg, qu, su, qd, sd,
                           out);
}

// oracle_layer with the tail skip at threshold tail_rank (0 = off).
int oracle_layer_tail(int H, int E, int k, int I, int R, int tail_rank, const float* router,
                      const uint16_t* x_bf16, int P, const int32_t* prov_ids, const int8_t* qg,
                      const uint16_t* sg, const int8_t* qu, const uint16_t* su, const int8_t* qd,
                      const uint16_t* sd, double* out) {
  if (I <= 0 || I % 32) return -1;
  Routing rt;
  if (route(H, E, k, R, router, x_bf16, rt, tail_rank)) return -1;
  Provided pv{P, prov_ids, qg, qu, qd, sg, su, sd};
  std::vector<int> slot(E, -1);
  for (int e : rt.uni) {
    slot[e] = pv.index_of(e);
    if (slot[e] < 0) return -2;
  }
  std::vector<float> x(H);
  std::vector<double> y(H);
  for (int r = 0; r < R; ++r) {
    for (int h = 0; h < H; ++h) x[h] = bf16_bits_to_float(x_bf16[(size_t)r * H + h]);
    double* o = out + (size_t)r * H;
    for (int h = 0; h < H; ++h) o[h] = 0.0;
    for (int j = 0; j < k; ++j) {
      if (!rt.keep[(size_t)r * k + j]) continue;
      int e = rt.ids[(size_t)r * k + j];
      ffn_of(H, I, pv, slot[e], x.data(), y.data());
      double wj = rt.w[(size_t)r * k + j];
      for (int h = 0; h < H; ++h) o[h] += wj * y[h];
    }
  }
  return 0;
}

// Brute-force dense evaluation: every one of the E experts (all provided, P == E,
// prov_ids == 0..E-1) runs for every row; the dense gate vector is w_j at the
// row's picks and 0 elsewhere; the combine runs over e ascending.
int oracle_layer_dense(int H, int E, int k, int I, int R, const float* router,
                       const uint16_t* x_bf16, const int8_t* qg, const uint16_t* sg,
                       const int8_t* qu, const uint16_t* su, const int8_t* qd,
                       const uint16_t* sd, double* out) {
  return oracle_layer_dense_tail(H, E, k, I, R, 0, router, x_bf16, qg, sg, qu, su, qd, sd, out);
}

// oracle_layer_dense with the tail skip (a dropped pick's gate entry stays 0).
int oracle_layer_dense_tail(int H, int E, int k, int I, int R, int tail_rank, const float* router,
                            const uint16_t* x_bf16, const int8_t* qg, const uint16_t* sg,
                            const int8_t* qu, const uint16_t* su, const int8_t* qd,
                            const uint16_t* sd, double* out) {
  if (I <= 0 || I % 32) return -1;
  Routing rt;
  if (route(H, E, k, R, router, x_bf16, rt, tail_rank)) return -1;
  std::vector<int32_t> all(E);
  for (int e = 0; e < E; ++e) all[e] = e;
  Provided pv{E, all.data(), qg, qu, qd, sg, su, sd};
  std::vector<float> x(H);
  std::vector<double> y(H), gate(E);
  for (int r = 0; r < R; ++r) {
    for (int h = 0; h < H; ++h) x[h] = bf16_bits_to_float(x_bf16[(size_t)r * H + h]);
    for (int e = 0; e < E; ++e) gate[e] = 0.0;
    for (int j = 0; j < k; ++j)
      if (rt.keep[(size_t)r * k + j]) gate[rt.ids[(size_t)r * k + j]] = rt.w[(size_t)r * k + j];
    double* o = out + (size_t)r * H;
    for (int h = 0; h < H; ++h) o[h] = 0.0;
    for (int e = 0; e < E; ++e) {
      ffn_of(H, I, pv, e, x.data(), y.data());
      for (int h = 0; h < H; ++h) o[h] += gate[e] * y[h];
    }
  }
  return 0;
}

// a4 + a5 for one (row, expert) pair: y[H] = Wd (silu(Wg x) * (Wu x)) in fp64, with
// x the row's bf16 activations; qg/qu [I][H], sg/su [I][H/32], qd [H][I], sd [H][I/32].
int oracle_expert_ffn(int H, int I, const uint16_t* x_bf16, const int8_t* qg, const uint16_t* sg,
                      const int8_t* qu, const uint16_t* su, const int8_t* qd, const uint16_t* sd,
                      double* y) {
  if (H <= 0 || H % 32 || I <= 0 || I % 32) return -1;
  std::vector<float> x(H);
  for (int h = 0; h < H; ++h) x[h] = bf16_bits_to_float(x_bf16[h]);
  expert_ffn(H, I, x.data(), qg, sg, qu, su, qd, sd, y);
  return 0;
}

// Unique expert bytes of a round: |U| experts, each 3 matrices of H*I int4 codes
// stored as 16 B of codes + 2 B fp16 scale per 32 codes.
int64_t oracle_unique_expert_bytes(int H, int I, int n_union) {
  return (int64_t)n_union * 3 * (int64_t)H * I / 32 * 18;
}

}  // extern "C"
