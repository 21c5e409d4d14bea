// GB300 (sm_103a) kernel and C ABI of the MoE layer of a speculative-decoding verify
// round.  See include/moe_verify.h for the operation and the contract.
//
// One persistent cooperative kernel (k_round, one CTA per SM) runs a whole round of L
// layers.  Per layer, with grid-wide barriers B1..B3 in between:
//   P1  router GEMV: one warp per expert, canonical fp32 order -> logits in the
//       workspace.  The next layer's router weights are prefetched into L2 while the
//       current layer streams its experts (they do not depend on any data).
//   B1
//   P2  every CTA reads the logits and builds the same routing in shared memory:
//       per-row top-k (warp per row, redux.sync selection, lower id wins ties),
//       renormalised weights, the ascending expert union U and, per union expert,
//       the (row, rank) pairs that picked it.
//   P3  split-K expert items, item = (union expert, 32-row slice of the intermediate
//       dimension), handed to CTAs round-robin.  Each CTA double-buffers items in
//       shared memory: one elected thread issues 1-D bulk TMA copies of the item's
//       gate/up rows + scales (mbarrier A) and the matching down K-block + scales
//       (mbarrier B); the CTA computes g, v, h = silu(g) v for each of the expert's
//       rows as soon as A lands, then the down partial Wd[:, slice] h[slice] once B
//       lands, and writes it per (row, rank, slice) to the workspace.
//   B2
//   P4  out[r][o] = sum_j w[r][j] * sum_s partial[r, j, s][o], a fixed order, so a
//       row's output depends only on that row (bitwise), whatever shares the round.
//   B3  (layer l+1's router waits for layer l's output, as a real decode would)
//
// Dequantisation without a convert instruction: a nibble n placed in bits [p, p+4) of
// an otherwise-zero fp32 word is the subnormal n * 2^(p-149); an fma with
// x * 2^(87-4m) (m = the nibble's slot) yields n * x * 2^-62 exactly.  One AND per
// weight (plus one shift per 8), and packed f32x2 FMAs over pairs of weights.  The
// code offset (q = n - 8) is applied once per 32-element block:
// sum (n-8) x = 2^62 acc - 8 sum x.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <vector>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int NT = 512;  // threads per CTA
constexpr int NW = NT / 32;
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
// device waits count SM cycles: 2 cycles per requested ns bounds the wall time between
// ns (at ~2 GHz) and a few times ns at lower clocks
constexpr long long kCyclesPerNs = 2;
constexpr long long kDefaultWaitCycles = (long long)kDefaultWaitNs * kCyclesPerNs;
constexpr int kPhases = 7;  // phase stamps per layer when profiling

struct LayerPtrs {
  const float* router;
  const uint8_t* gu_nib;
  const uint16_t* gu_sc;
  const uint8_t* dn_nib;
  const uint16_t* dn_sc;
};

struct RoundArgs {
  int H, E, k, I, R, L;
  int route_only;
  const uint16_t* x;  // [L][R][H] bf16 bits
  float* out;         // [L][R][H]
  int* stats;         // [L] |U| per layer, or null
  unsigned* bar;      // [0] barrier arrivals, [1] abort flag
  float* logits;      // [R][E]
  float* partial;     // [R*k][I/32][H]
  int* user_ids;      // moe_route outputs (CTA 0 writes them)
  float* user_w;
  int* user_union;
  int* user_nunion;
  unsigned* status;
  long long wait_cycles;
  long long* phase_ts;  // [L][kPhases][grid] globaltimer stamps, or null
  LayerPtrs layer[kMaxLayers];
};

// ---------------------------------------------------------------------------------
// device helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ long long gtimer() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(phase)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(phase)
      : "memory");
  return ok != 0;
}

// Waits for `phase` of the mbarrier for at most `limit` SM cycles; on giving up it
// raises the timeout bit of the status word and returns false.  The first poll does
// not block, so a bound of a few cycles gives up deterministically.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t phase, unsigned* status,
                                                  long long limit) {
  const long long t0 = clock64();
  if (mbar_test_wait(bar, phase)) return true;
  while (true) {
    if (clock64() - t0 > limit) {
      atomicOr(status, kStatusTimeout);
      return false;
    }
    if (mbar_try_wait(bar, phase)) return true;
  }
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// packed pairs of fp32 for fma.rn.f32x2
typedef unsigned long long f2_t;

__device__ __forceinline__ f2_t f2pack(float lo, float hi) {
  f2_t r;
  asm("mov.b64 %0, {%1,%2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ float f2sum(f2_t v) {
  float lo, hi;
  asm("mov.b64 {%0,%1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return __fadd_rn(lo, hi);
}

__device__ __forceinline__ void ffma2(f2_t& acc, f2_t a, f2_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// 2^(87 - 4m) for nibble slots m = 0..4 and 2^(99 - 4m) for m = 5..7 (those three are
// read after a 12-bit right shift): the factor that turns the subnormal n * 2^e_m into
// n * x * 2^-62 under an fma.
__device__ __forceinline__ float slot_scale(int m) {
  const int e = (m <= 4) ? 87 - 4 * m : 99 - 4 * m;
  return __int_as_float((127 + e) << 23);
}

// acc += the 8 nibbles of w times xs[4] (pre-scaled pairs), slot pairs (0,1) (2,3) (4,5) (6,7)
__device__ __forceinline__ void dot8x2(uint32_t w, const f2_t* xs, f2_t& acc) {
  const uint32_t t = w >> 12;
  ffma2(acc, f2pack(__uint_as_float(w & 0x0000000Fu), __uint_as_float(w & 0x000000F0u)), xs[0]);
  ffma2(acc, f2pack(__uint_as_float(w & 0x00000F00u), __uint_as_float(w & 0x0000F000u)), xs[1]);
  ffma2(acc, f2pack(__uint_as_float(w & 0x000F0000u), __uint_as_float(t & 0x00000F00u)), xs[2]);
  ffma2(acc, f2pack(__uint_as_float(t & 0x0000F000u), __uint_as_float(t & 0x000F0000u)), xs[3]);
}

// 2^-62 * sum_{k<32} n_k x_k for one 16-byte block of codes; xs = 16 pre-scaled pairs.
__device__ __forceinline__ float dot32(const uint4 nb, const f2_t* xs) {
  f2_t a0 = 0ull, a1 = 0ull;
  dot8x2(nb.x, xs + 0, a0);
  dot8x2(nb.y, xs + 4, a1);
  dot8x2(nb.z, xs + 8, a0);
  dot8x2(nb.w, xs + 12, a1);
  return __fadd_rn(f2sum(a0), f2sum(a1));
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ float half_bits(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// float -> unsigned key with the same order; -0 is first folded into +0 so that a
// signed-zero pair ties (and the lower id wins), as the definition asks.
__device__ __forceinline__ unsigned order_key(float v) {
  const unsigned u = __float_as_uint(__fadd_rn(v, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// ---------------------------------------------------------------------------------
// grid barrier (all CTAs are co-resident: cooperative launch, one CTA per SM)

struct Sync {
  unsigned epoch = 0;
};

// Returns false if the round must be abandoned (a CTA gave up somewhere).
__device__ bool grid_sync(const RoundArgs& a, Sync& sy) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    sy.epoch += 1;
    const unsigned target = sy.epoch * gridDim.x;
    __threadfence();
    atomicAdd(a.bar, 1u);
    int ok = 1;
    const long long t0 = clock64();
    while (ld_acquire(a.bar) < target) {
      if (ld_relaxed(a.bar + 1)) {
        ok = 0;
        break;
      }
      if (clock64() - t0 > a.wait_cycles) {
        atomicOr(a.status, kStatusTimeout);
        atomicExch(a.bar + 1, 1u);
        ok = 0;
        break;
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

__device__ __forceinline__ void stamp(const RoundArgs& a, int l, int ph) {
  if (a.phase_ts && threadIdx.x == 0)
    a.phase_ts[((size_t)l * kPhases + ph) * gridDim.x + blockIdx.x] = gtimer();
}

// ---------------------------------------------------------------------------------
// P1: router logits, one warp per expert, canonical order

// Lane l accumulates elements 128c + 4l + j for c ascending.  The c-loop runs in groups
// of 8 (32 weights per lane in registers); for H > 1024 each lane's partial of every
// row is carried between groups in `carry` (idle staging memory), so the order of the
// fmas is exactly the canonical one.
__device__ void router_phase(const RoundArgs& a, const float* router, const uint16_t* x,
                             float* carry_all) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int NC = a.H >> 7;  // <= 16
  const int gw = blockIdx.x * NW + warp;
  float* carry = carry_all + (size_t)warp * a.R * 32;
  for (int e = gw; e < a.E; e += gridDim.x * NW) {
    const float4* wr = reinterpret_cast<const float4*>(router + (size_t)e * a.H) + lane;
    for (int g = 0; g < NC; g += 8) {
      float4 wv[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        if (g + c < NC) wv[c] = __ldg(wr + 32 * (g + c));
      const bool last = g + 8 >= NC;
      for (int r = 0; r < a.R; ++r) {
        const uint2* xr = reinterpret_cast<const uint2*>(x + (size_t)r * a.H) + lane;
        float p = (g == 0) ? 0.f : carry[r * 32 + lane];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          if (g + c < NC) {
            const uint2 xv = __ldg(xr + 32 * (g + c));
            p = __fmaf_rn(wv[c].x, bf16_lo(xv.x), p);
            p = __fmaf_rn(wv[c].y, bf16_hi(xv.x), p);
            p = __fmaf_rn(wv[c].z, bf16_lo(xv.y), p);
            p = __fmaf_rn(wv[c].w, bf16_hi(xv.y), p);
          }
        }
        if (!last) {
          carry[r * 32 + lane] = p;
        } else {
          p = warp_sum(p);
          if (lane == 0) a.logits[(size_t)r * a.E + e] = p;
        }
      }
      __syncwarp();
    }
  }
}

// ---------------------------------------------------------------------------------
// P2: routing tables of one layer, built by every CTA in its shared memory

struct Tables {
  int* uni;      // [E] ascending union
  int* csr_off;  // [E+1] offsets into pair
  int* pair;     // [R*k] pair index p = r*k + j, grouped by union expert, rows ascending
  float* w;      // [R*k] renormalised weight of pair p
  int* n_union;  // [1]
};

// scratch (inside the staging area, free while routing): mask [E], off_e [E], ids [R*k]
__device__ int route_phase(const RoundArgs& a, const Tables& T, unsigned* s_mask, int* s_off_e,
                           int* s_ids, int layer) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, k = a.k, R = a.R;
  for (int e = tid; e < E; e += NT) s_mask[e] = 0u;
  const int NE = (E + 31) >> 5;  // <= 32
  for (int r = warp; r < R; r += NW) {
    unsigned key[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      if (t < NE) {
        const int e = lane + 32 * t;
        key[t] = (e < E) ? order_key(__ldcg(a.logits + (size_t)r * E + e)) : 0u;
      }
    }
    float my_l = 0.f;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
      unsigned bk = 0u;
      int bt = 0;
#pragma unroll
      for (int t = 0; t < 32; ++t)
        if (t < NE && key[t] > bk) {  // strict: the first (lowest id) of equal keys stays
          bk = key[t];
          bt = t;
        }
      const unsigned m = __reduce_max_sync(0xffffffffu, bk);
      const unsigned cand = (bk == m && m != 0u) ? (unsigned)(lane + 32 * bt) : 0xffffffffu;
      const unsigned win = __reduce_min_sync(0xffffffffu, cand);
      if ((int)(win & 31u) == lane) {
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (t == (int)(win >> 5)) key[t] = 0u;
      }
      if (lane == j) {
        my_l = key_value(m);
        my_id = (int)win;
      }
    }
    // weights: exp(l_j - l_1) / sum over the k picks, summed in rank order
    const float l1 = __shfl_sync(0xffffffffu, my_l, 0);
    const float ex = (lane < k) ? expf(my_l - l1) : 0.f;
    float den = 0.f;
    for (int j = 0; j < k; ++j) den = __fadd_rn(den, __shfl_sync(0xffffffffu, ex, j));
    if (lane < k) {
      const float wj = __fdiv_rn(ex, den);
      const int p = r * k + lane;
      s_ids[p] = my_id;
      T.w[p] = wj;
      if (blockIdx.x == 0) {
        if (a.user_ids) a.user_ids[p] = my_id;
        if (a.user_w) a.user_w[p] = wj;
      }
    }
  }
  __syncthreads();
  for (int p = tid; p < R * k; p += NT) atomicOr(&s_mask[s_ids[p]], 1u << (p / k));
  __syncthreads();

  // exclusive scans over e of (picked ? 1 : 0) and popc(mask): union index, pair offset
  __shared__ int s_wf[NW], s_wc[NW];
  const int per = (E + NT - 1) / NT;
  const int e0 = tid * per;
  int lf = 0, lc = 0;
  for (int e = e0; e < e0 + per && e < E; ++e) {
    const unsigned m = s_mask[e];
    lf += (m != 0u);
    lc += __popc(m);
  }
  int incf = lf, incc = lc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int tf = __shfl_up_sync(0xffffffffu, incf, o);
    const int tc = __shfl_up_sync(0xffffffffu, incc, o);
    if (lane >= o) {
      incf += tf;
      incc += tc;
    }
  }
  if (lane == 31) {
    s_wf[warp] = incf;
    s_wc[warp] = incc;
  }
  __syncthreads();
  int basef = incf - lf, basec = incc - lc;
  for (int w2 = 0; w2 < warp; ++w2) {
    basef += s_wf[w2];
    basec += s_wc[w2];
  }
  for (int e = e0; e < e0 + per && e < E; ++e) {
    const unsigned m = s_mask[e];
    if (m) {
      s_off_e[e] = basec;
      T.uni[basef] = e;
      T.csr_off[basef] = basec;
      if (blockIdx.x == 0 && a.user_union) a.user_union[basef] = e;
      ++basef;
      basec += __popc(m);
    }
  }
  if (tid == NT - 1) {
    // the last thread's running totals are the union size and the pair count
    *T.n_union = basef;
    T.csr_off[basef] = basec;
    if (blockIdx.x == 0) {
      if (a.user_nunion) *a.user_nunion = basef;
      if (a.stats) a.stats[layer] = basef;
    }
  }
  __syncthreads();
  for (int p = tid; p < R * k; p += NT) {
    const int e = s_ids[p], r = p / k;
    T.pair[s_off_e[e] + __popc(s_mask[e] & ((1u << r) - 1u))] = p;
  }
  __syncthreads();
  return *T.n_union;
}

// ---------------------------------------------------------------------------------
// P3: expert items

// one staged item: gate/up codes 32H, gate/up scales 4H, down codes 16H, down scales 2H
__host__ __device__ constexpr size_t stage_bytes(int H) { return (size_t)54 * H; }

struct Stage {
  uint8_t* base;
  uint32_t bar_a, bar_b;
};

__device__ void issue_item(const RoundArgs& a, const LayerPtrs& W, const Stage& st, int u, int s) {
  const size_t H = (size_t)a.H, I = (size_t)a.I, NB = H / 32;
  // order earlier generic-proxy accesses of this buffer before the async-proxy writes
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(st.bar_a, (uint32_t)(36 * H));
  bulk_g2s(smem_u32(st.base), W.gu_nib + (size_t)u * I * H + (size_t)s * 32 * H, (uint32_t)(32 * H),
           st.bar_a);
  bulk_g2s(smem_u32(st.base + 32 * H), W.gu_sc + (size_t)u * (I * H / 16) + (size_t)s * 64 * NB,
           (uint32_t)(4 * H), st.bar_a);
  mbar_expect_tx(st.bar_b, (uint32_t)(18 * H));
  bulk_g2s(smem_u32(st.base + 36 * H), W.dn_nib + (size_t)u * (I * H / 2) + (size_t)s * 16 * H,
           (uint32_t)(16 * H), st.bar_b);
  bulk_g2s(smem_u32(st.base + 52 * H), W.dn_sc + (size_t)u * (I * H / 32) + (size_t)s * H,
           (uint32_t)(2 * H), st.bar_b);
}

// Computes one staged item for every row of its expert.  Returns false on a timeout.
// Stage b's state lives in two bitfields: `ph` holds the parity to wait for (bit 2b:
// gate/up barrier A, bit 2b+1: down barrier B) and `pend` marks copies in flight.  On
// success both barriers have been consumed (parities flipped, pending bits cleared);
// on failure `pend` still marks the copies the caller must drain.
template <int NBL>
__device__ bool compute_item(const RoundArgs& a, const Tables& T, const Stage& st, int b,
                             unsigned& ph, unsigned& pend, int ui, int s, const uint16_t* x,
                             float* s_gv, float* s_h, float* s_hsum) {
  const int H = a.H, NB = H >> 5, NS = a.I >> 5;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint8_t* s_gu = st.base;
  const uint16_t* s_gus = reinterpret_cast<const uint16_t*>(st.base + 32 * (size_t)H);
  const uint8_t* s_dn = st.base + 36 * (size_t)H;
  const uint16_t* s_dns = reinterpret_cast<const uint16_t*>(st.base + 52 * (size_t)H);

  const unsigned bit_a = 1u << (2 * b), bit_b = 2u << (2 * b);
  bool ok = mbar_wait_bounded(st.bar_a, (ph & bit_a) ? 1u : 0u, a.status, a.wait_cycles);
  if (__syncthreads_or(!ok)) return false;
  ph ^= bit_a;
  pend &= ~bit_a;
  bool have_b = false;
  const int p0 = T.csr_off[ui], p1 = T.csr_off[ui + 1];
  for (int pp = p0; pp < p1; ++pp) {
    const int pair = T.pair[pp];
    const int r = pair / a.k;
    // ---- gate / up: warp per weight row, lane per 32-element block ----
    // 64 weight rows (32 gate, 32 up) over NW warps; the lane's blocks are visited one
    // at a time so only one block of pre-scaled activations sits in registers.
    constexpr int RPW = 64 / NW;
    float part[RPW];
#pragma unroll
    for (int q = 0; q < RPW; ++q) part[q] = 0.f;
#pragma unroll
    for (int t = 0; t < NBL; ++t) {
      const int blk = lane + 32 * t;
      if (blk < NB) {
        f2_t xs[16];
        float sum = 0.f;
        const uint4* xp = reinterpret_cast<const uint4*>(x + (size_t)r * H + 32 * blk);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = __ldg(xp + q);
          const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int z = 0; z < 4; ++z) {
            const float lo = bf16_lo(wds[z]), hi = bf16_hi(wds[z]);
            const int k0 = 8 * q + 2 * z;  // element index in the block; slots k0&7, +1
            xs[k0 >> 1] = f2pack(lo * slot_scale(k0 & 7), hi * slot_scale((k0 + 1) & 7));
            sum = __fadd_rn(sum, lo);
            sum = __fadd_rn(sum, hi);
          }
        }
        const float xsum8 = -8.f * sum;
#pragma unroll
        for (int q = 0; q < RPW; ++q) {
          const int wr = warp + NW * q;
          const uint4 nb = *reinterpret_cast<const uint4*>(s_gu + ((size_t)wr * NB + blk) * 16);
          const float sc = half_bits(s_gus[wr * NB + blk]);
          const float acc = dot32(nb, xs);
          part[q] = __fmaf_rn(sc, __fmaf_rn(acc, 0x1p62f, xsum8), part[q]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < RPW; ++q) {
      const float v = warp_sum(part[q]);
      if (lane == 0) s_gv[warp + NW * q] = v;
    }
    __syncthreads();
    // ---- SwiGLU on the slice's 32 intermediate rows ----
    if (warp == 0) {
      const float g = s_gv[lane], v = s_gv[32 + lane];
      const float hh = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.f, expf(-g))), v);
      s_h[lane] = hh * slot_scale(lane & 7);
      const float hs = warp_sum(hh);
      if (lane == 0) *s_hsum = -8.f * hs;
    }
    if (!have_b) {
      ok = mbar_wait_bounded(st.bar_b, (ph & bit_b) ? 1u : 0u, a.status, a.wait_cycles);
      if (__syncthreads_or(!ok)) return false;
      ph ^= bit_b;
      pend &= ~bit_b;
      have_b = true;
    } else {
      __syncthreads();
    }
    // ---- down partial: thread per output row, one 32-element K-block each ----
    f2_t hreg[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) hreg[q] = f2pack(s_h[2 * q], s_h[2 * q + 1]);
    const float hsum8 = *s_hsum;
    float* dst = a.partial + ((size_t)pair * NS + s) * H;
    for (int o = tid; o < H; o += NT) {
      const uint4 nb = *reinterpret_cast<const uint4*>(s_dn + (size_t)o * 16);
      const float sc = half_bits(s_dns[o]);
      const float acc = dot32(nb, hreg);
      dst[o] = __fmul_rn(sc, __fmaf_rn(acc, 0x1p62f, hsum8));
    }
    // the next row's gate/up may overwrite s_gv only after everyone has read s_h
    __syncthreads();
  }
  if (!have_b) {  // (every union expert has a row, so this only keeps phases paired)
    ok = mbar_wait_bounded(st.bar_b, (ph & bit_b) ? 1u : 0u, a.status, a.wait_cycles);
    if (__syncthreads_or(!ok)) return false;
    ph ^= bit_b;
    pend &= ~bit_b;
  }
  return true;
}

// ---------------------------------------------------------------------------------
// P4: fixed-order weighted reduction of the partials into the layer output

__device__ void reduce_phase(const RoundArgs& a, const Tables& T, float* out) {
  const int H = a.H, k = a.k, NS = a.I >> 5;
  int kp = 1;
  while (kp < k) kp <<= 1;  // lanes per output; kp divides 32
  const int lane = threadIdx.x & 31;
  const int gbase = lane & ~(kp - 1);
  const long long total = (long long)a.R * H * kp;
  for (long long t = (long long)blockIdx.x * NT + threadIdx.x; t < total;
       t += (long long)gridDim.x * NT) {
    const int j = (int)(t & (kp - 1));
    const long long ro = t / kp;
    const int r = (int)(ro / H), o = (int)(ro - (long long)r * H);
    float y = 0.f;
    if (j < k) {
      const float* src = a.partial + (size_t)(r * k + j) * NS * H + o;
      for (int s = 0; s < NS; ++s) y = __fadd_rn(y, __ldcg(src + (size_t)s * H));
    }
    float acc = 0.f;
    for (int jj = 0; jj < k; ++jj) {
      const float yj = __shfl_sync(0xffffffffu, y, gbase + jj);
      acc = __fmaf_rn(T.w[r * k + jj], yj, acc);
    }
    if (j == 0) out[(size_t)r * H + o] = acc;
  }
}

// ---------------------------------------------------------------------------------
// shared-memory plan

struct SmemPlan {
  size_t stage, stage0, stage1, bars, gv, uni, csr, pair, w, nunion, total;
};

__host__ __device__ inline size_t up128(size_t x) { return (x + 127) & ~(size_t)127; }

__host__ __device__ inline SmemPlan smem_plan(int H, int E, int R, int k) {
  SmemPlan p{};
  p.stage = up128(stage_bytes(H));
  size_t off = 0;
  p.stage0 = off;  off += p.stage;
  p.stage1 = off;  off += p.stage;
  p.bars = off;    off += 64;
  p.gv = off;      off += up128((64 + 32 + 4) * 4);
  p.uni = off;     off += up128((size_t)E * 4);
  p.csr = off;     off += up128((size_t)(E + 1) * 4);
  p.pair = off;    off += up128((size_t)R * k * 4);
  p.w = off;       off += up128((size_t)R * k * 4);
  p.nunion = off;  off += 128;
  p.total = off;
  return p;
}

template <int NBL>
__global__ void __launch_bounds__(NT, 1) k_round(const __grid_constant__ RoundArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x;
  const SmemPlan P = smem_plan(a.H, a.E, a.R, a.k);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bars);
  // stage b: buffer at stage0 + b * stage, barriers bars[2b] (A) and bars[2b + 1] (B)
  auto stage_of = [&](int b) {
    return Stage{smem + P.stage0 + (size_t)b * P.stage, smem_u32(bars + 2 * b),
                 smem_u32(bars + 2 * b + 1)};
  };
  float* s_gv = reinterpret_cast<float*>(smem + P.gv);
  float* s_h = s_gv + 64;
  float* s_hsum = s_h + 32;
  Tables T{reinterpret_cast<int*>(smem + P.uni), reinterpret_cast<int*>(smem + P.csr),
           reinterpret_cast<int*>(smem + P.pair), reinterpret_cast<float*>(smem + P.w),
           reinterpret_cast<int*>(smem + P.nunion)};
  // routing scratch lives in the (then idle) staging area
  unsigned* s_mask = reinterpret_cast<unsigned*>(smem + P.stage0);
  int* s_off_e = reinterpret_cast<int*>(smem + P.stage0 + (size_t)a.E * 4);
  int* s_ids = reinterpret_cast<int*>(smem + P.stage0 + (size_t)a.E * 8);
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(bars + i), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  Sync sy;
  unsigned ph = 0u;    // parity to wait for: bit 2b = stage b's barrier A, bit 2b+1 = B
  unsigned pend = 0u;  // copies in flight, same bit layout
  const int G = gridDim.x, NS = a.I >> 5;
  const size_t RH = (size_t)a.R * a.H;
  for (int l = 0; l < a.L; ++l) {
    const LayerPtrs& W = a.layer[l];
    const uint16_t* x = a.x + (size_t)l * RH;
    stamp(a, l, 0);
    router_phase(a, W.router, x, reinterpret_cast<float*>(smem + P.stage0));
    stamp(a, l, 1);
    if (!grid_sync(a, sy)) return;  // B1: all logits written
    stamp(a, l, 2);
    const int U = route_phase(a, T, s_mask, s_off_e, s_ids, l);
    stamp(a, l, 3);
    if (a.route_only) return;
    const int n_items = U * NS;
    for (int n = 0; n < 2; ++n) {
      const int it = blockIdx.x + n * G;
      if (it < n_items) {
        pend |= 3u << (2 * n);  // every thread tracks what thread 0 issues
        if (tid == 0) issue_item(a, W, stage_of(n), T.uni[it / NS], it % NS);
      }
    }
    if (tid == 0) {
      if (l + 1 < a.L) {  // the next layer's router weights do not depend on any data
        const size_t bytes = (size_t)a.E * a.H * 4;
        const size_t chunk = ((bytes / G) + 15) & ~(size_t)15;
        const size_t b0 = (size_t)blockIdx.x * chunk;
        if (b0 < bytes) {
          const size_t n = (bytes - b0 < chunk) ? bytes - b0 : chunk;
          prefetch_l2(reinterpret_cast<const char*>(a.layer[l + 1].router) + b0, (uint32_t)n);
        }
      }
    }
    for (int n = 0;; ++n) {
      const int it = blockIdx.x + n * G;
      if (it >= n_items) break;
      const int b = n & 1;
      if (!compute_item<NBL>(a, T, stage_of(b), b, ph, pend, it / NS, it % NS, x, s_gv, s_h,
                             s_hsum)) {
        // give every copy still in flight a bounded chance to land, then leave
        for (int q = 0; q < 4; ++q)
          if (pend & (1u << q))
            mbar_wait_bounded(smem_u32(bars + q), (ph >> q) & 1u, a.status, kDefaultWaitCycles);
        if (tid == 0) atomicExch(a.bar + 1, 1u);
        return;
      }
      // compute_item ends with a CTA barrier: the stage is free again
      const int nxt = it + 2 * G;
      if (nxt < n_items) {
        pend |= 3u << (2 * b);
        if (tid == 0) issue_item(a, W, stage_of(b), T.uni[nxt / NS], nxt % NS);
      }
    }
    stamp(a, l, 4);
    if (!grid_sync(a, sy)) return;  // B2: all partials written
    stamp(a, l, 5);
    reduce_phase(a, T, a.out + (size_t)l * RH);
    stamp(a, l, 6);
    if (l + 1 < a.L && !grid_sync(a, sy)) return;  // B3: layer output complete
  }
}

}  // namespace
}  // namespace moe

// =====================================================================================
// host side

using namespace moe;

struct GraphKey {
  std::vector<moe_layer_w> layers;
  int32_t rows = 0;
  const void *x = nullptr, *out = nullptr, *stats = nullptr, *ws = nullptr, *stream = nullptr;
  size_t ws_bytes = 0;
  bool operator==(const GraphKey& o) const {
    if (rows != o.rows || x != o.x || out != o.out || stats != o.stats || ws != o.ws ||
        stream != o.stream || ws_bytes != o.ws_bytes || layers.size() != o.layers.size())
      return false;
    return layers.empty() ||
           std::memcmp(layers.data(), o.layers.data(), layers.size() * sizeof(moe_layer_w)) == 0;
  }
};

struct moe_handle {
  moe_dims dims;
  int device = 0;
  int sm_count = 0;
  unsigned* status = nullptr;
  unsigned long long wait_ns = kDefaultWaitNs;
  int32_t last_launches = 0;
  GraphKey gkey;
  cudaGraphExec_t gexec = nullptr;
  int32_t graph_launches = 0;
  // profiling of eager calls (moe_profile): event pairs and phase stamps
  bool profiling = false;
  std::vector<cudaEvent_t> ev;  // start/stop pairs
  size_t ev_used = 0;
  long long* phase_ts = nullptr;  // [kMaxLayers][kPhases][sm_count]
  int32_t phase_layers = 0;
};

namespace {

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      prev = -1;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int nbl_of(int H) { return (H + 1023) / 1024; }

int check_layer(const moe_layer_w* w) {
  if (!w) return MOE_EINVAL;
  if (!aligned16(w->router) || !aligned16(w->gateup_nib) || !aligned16(w->gateup_scale) ||
      !aligned16(w->down_nib) || !aligned16(w->down_scale))
    return MOE_EINVAL;
  return MOE_OK;
}

size_t smem_bytes(const moe_dims& d, int rows) {
  return smem_plan(d.hidden, d.n_experts, rows, d.top_k).total;
}

void fill_args(RoundArgs& a, const moe_handle* h, int rows, void* ws) {
  const moe_dims& d = h->dims;
  const WsLayout L = ws_layout(d, rows);
  char* base = static_cast<char*>(ws);
  a.H = d.hidden;
  a.E = d.n_experts;
  a.k = d.top_k;
  a.I = d.inter;
  a.R = rows;
  a.bar = reinterpret_cast<unsigned*>(base + L.ctrl);
  a.logits = reinterpret_cast<float*>(base + L.logits);
  a.partial = reinterpret_cast<float*>(base + L.partial);
  a.status = h->status;
  const unsigned long long ns = h->wait_ns < (1ull << 40) ? h->wait_ns : (1ull << 40);
  a.wait_cycles = (long long)ns * kCyclesPerNs;
}

cudaError_t launch_round(moe_handle* h, const RoundArgs& a, cudaStream_t st, bool capturing) {
  cudaError_t e = cudaMemsetAsync(a.bar, 0, 256, st);
  if (e != cudaSuccess) return e;
  const bool prof = h->profiling && !capturing;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (prof) {
    while (h->ev.size() < h->ev_used + 2) {
      cudaEvent_t ev;
      if (cudaEventCreate(&ev) != cudaSuccess) return cudaGetLastError();
      h->ev.push_back(ev);
    }
    e0 = h->ev[h->ev_used];
    e1 = h->ev[h->ev_used + 1];
    h->ev_used += 2;
    cudaEventRecord(e0, st);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(h->sm_count);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem_bytes(h->dims, a.R);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (nbl_of(a.H) == 1)
    e = cudaLaunchKernelEx(&cfg, k_round<1>, a);
  else
    e = cudaLaunchKernelEx(&cfg, k_round<2>, a);
  if (prof) cudaEventRecord(e1, st);
  return e;
}

int common_checks(moe_handle* h, const uint16_t* x, int32_t rows, void* ws, size_t ws_bytes) {
  if (!h || !aligned16(x) || !ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_EINVAL;
  if (rows < 1 || rows > h->dims.max_rows) return MOE_EINVAL;
  if (ws_bytes < ws_layout(h->dims, rows).total) return MOE_EWORKSPACE;
  return MOE_OK;
}

void copy_layers(RoundArgs& a, const moe_layer_w* layers, int32_t L) {
  for (int32_t l = 0; l < L; ++l) {
    a.layer[l].router = layers[l].router;
    a.layer[l].gu_nib = layers[l].gateup_nib;
    a.layer[l].gu_sc = layers[l].gateup_scale;
    a.layer[l].dn_nib = layers[l].down_nib;
    a.layer[l].dn_sc = layers[l].down_scale;
  }
}

}  // namespace

extern "C" {

int moe_create(const moe_dims* dims, int device, moe_handle** out) {
  if (!out) return MOE_EINVAL;
  *out = nullptr;
  int rc = check_dims(dims);
  if (rc != MOE_OK) return rc;
  const size_t smem = smem_bytes(*dims, dims->max_rows);
  if (smem > 227 * 1024) return MOE_EUNSUPPORTED;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  DeviceGuard g(device);
  if (!g.ok) return MOE_ECUDA;
  int coop = 0;
  moe_handle* h = new moe_handle();
  h->dims = *dims;
  h->device = device;
  if (cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device) != cudaSuccess || !coop ||
      cudaMalloc(&h->status, sizeof(unsigned)) != cudaSuccess ||
      cudaMemset(h->status, 0, sizeof(unsigned)) != cudaSuccess) {
    cudaGetLastError();
    if (h->status) cudaFree(h->status);
    delete h;
    return MOE_ECUDA;
  }
  cudaError_t e;
  int occ = 0;
  if (nbl_of(dims->hidden) == 1) {
    e = cudaFuncSetAttribute(k_round<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_round<1>, NT, smem);
  } else {
    e = cudaFuncSetAttribute(k_round<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_round<2>, NT, smem);
  }
  if (e != cudaSuccess || occ < 1) {
    cudaGetLastError();
    cudaFree(h->status);
    delete h;
    return MOE_ECUDA;
  }
  *out = h;
  return MOE_OK;
}

void moe_destroy(moe_handle* h) {
  if (!h) return;
  DeviceGuard g(h->device);
  if (h->gexec) cudaGraphExecDestroy(h->gexec);
  if (h->status) cudaFree(h->status);
  if (h->phase_ts) cudaFree(h->phase_ts);
  for (cudaEvent_t e : h->ev) cudaEventDestroy(e);
  delete h;
}

int moe_set_wait_limit_ns(moe_handle* h, uint64_t ns) {
  if (!h) return MOE_EINVAL;
  h->wait_ns = ns ? ns : kDefaultWaitNs;
  return MOE_OK;
}

int moe_route(moe_handle* h, const moe_layer_w* w, const uint16_t* x_bf16, int32_t rows,
              int32_t* topk_ids, float* topk_w, int32_t* union_ids, int32_t* n_union, void* ws,
              size_t ws_bytes, void* stream) {
  int rc = common_checks(h, x_bf16, rows, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  if (!w || !aligned16(w->router)) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  RoundArgs a{};
  fill_args(a, h, rows, ws);
  a.L = 1;
  a.route_only = 1;
  a.x = x_bf16;
  a.user_ids = topk_ids;
  a.user_w = topk_w;
  a.user_union = union_ids;
  a.user_nunion = n_union;
  a.layer[0].router = w->router;
  h->last_launches = 1;
  return launch_round(h, a, static_cast<cudaStream_t>(stream), false) == cudaSuccess ? MOE_OK
                                                                                    : MOE_ECUDA;
}

int moe_decode_layer(moe_handle* h, const moe_layer_w* w, const uint16_t* x_bf16, int32_t rows,
                     float* out, void* ws, size_t ws_bytes, void* stream) {
  int rc = common_checks(h, x_bf16, rows, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  if ((rc = check_layer(w)) != MOE_OK) return rc;
  if (!aligned16(out)) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  RoundArgs a{};
  fill_args(a, h, rows, ws);
  a.L = 1;
  a.x = x_bf16;
  a.out = out;
  copy_layers(a, w, 1);
  h->last_launches = 1;
  return launch_round(h, a, static_cast<cudaStream_t>(stream), false) == cudaSuccess ? MOE_OK
                                                                                    : MOE_ECUDA;
}

int moe_round(moe_handle* h, const moe_layer_w* layers, int32_t L, const uint16_t* x_bf16,
              int32_t rows, float* out, int32_t* stats, void* ws, size_t ws_bytes, int use_graph,
              void* stream) {
  int rc = common_checks(h, x_bf16, rows, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  if (!layers || L < 1 || !aligned16(out)) return MOE_EINVAL;
  if (L > kMaxLayers) return MOE_EUNSUPPORTED;
  for (int32_t l = 0; l < L; ++l)
    if ((rc = check_layer(&layers[l])) != MOE_OK) return rc;
  if (use_graph && !stream) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RoundArgs a{};
  fill_args(a, h, rows, ws);
  a.L = L;
  a.x = x_bf16;
  a.out = out;
  a.stats = stats;
  copy_layers(a, layers, L);
  if (!use_graph) {
    if (h->profiling && h->phase_ts) {
      a.phase_ts = h->phase_ts;
      h->phase_layers = L;
    }
    h->last_launches = 1;
    return launch_round(h, a, st, false) == cudaSuccess ? MOE_OK : MOE_ECUDA;
  }
  GraphKey key;
  key.layers.assign(layers, layers + L);
  key.rows = rows;
  key.x = x_bf16;
  key.out = out;
  key.stats = stats;
  key.ws = ws;
  key.stream = stream;
  key.ws_bytes = ws_bytes;
  if (!h->gexec || !(key == h->gkey)) {
    if (h->gexec) {
      cudaGraphExecDestroy(h->gexec);
      h->gexec = nullptr;
    }
    if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
      return MOE_ECUDA;
    cudaError_t e = launch_round(h, a, st, true);
    cudaGraph_t graph = nullptr;
    cudaError_t e2 = cudaStreamEndCapture(st, &graph);
    if (e != cudaSuccess || e2 != cudaSuccess || !graph) {
      if (graph) cudaGraphDestroy(graph);
      cudaGetLastError();
      return MOE_ECUDA;
    }
    e = cudaGraphInstantiate(&h->gexec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
      h->gexec = nullptr;
      cudaGetLastError();
      return MOE_ECUDA;
    }
    h->gkey = key;
    h->graph_launches = 1;
  }
  if (cudaGraphLaunch(h->gexec, st) != cudaSuccess) return MOE_ECUDA;
  h->last_launches = h->graph_launches;
  return MOE_OK;
}

int moe_last_device_status(moe_handle* h, void* stream) {
  if (!h) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  unsigned v = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ECUDA;
  if (cudaMemcpy(&v, h->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ECUDA;
  if (cudaMemset(h->status, 0, sizeof(unsigned)) != cudaSuccess) return MOE_ECUDA;
  return (v & kStatusTimeout) ? MOE_ETIMEOUT : MOE_OK;
}

int32_t moe_last_launch_count(const moe_handle* h) { return h ? h->last_launches : 0; }

int moe_profile(moe_handle* h, int enable) {
  if (!h) return MOE_EINVAL;
  h->profiling = enable != 0;
  h->ev_used = 0;
  h->phase_layers = 0;
  if (h->profiling && !h->phase_ts) {
    DeviceGuard g(h->device);
    if (!g.ok) return MOE_ECUDA;
    const size_t n = (size_t)kMaxLayers * kPhases * h->sm_count;
    if (cudaMalloc(&h->phase_ts, n * sizeof(long long)) != cudaSuccess) {
      cudaGetLastError();
      h->phase_ts = nullptr;
      return MOE_ECUDA;
    }
  }
  return MOE_OK;
}

int moe_profile_read(moe_handle* h, int kind, double* total_ms, int32_t* launches) {
  if (!h || !total_ms || !launches || kind != 0) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  double t = 0.0;
  int32_t n = 0;
  for (size_t i = 0; i + 1 < h->ev_used; i += 2) {
    if (cudaEventSynchronize(h->ev[i + 1]) != cudaSuccess) return MOE_ECUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, h->ev[i], h->ev[i + 1]) != cudaSuccess) return MOE_ECUDA;
    t += ms;
    ++n;
  }
  *total_ms = t;
  *launches = n;
  return MOE_OK;
}

int moe_profile_phases(moe_handle* h, double* mean_us, double* max_us, int32_t n_phases) {
  if (!h || !mean_us || !max_us || n_phases < kPhases - 1) return MOE_EINVAL;
  if (!h->phase_ts || h->phase_layers < 1) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  const int G = h->sm_count, L = h->phase_layers;
  std::vector<long long> ts((size_t)L * kPhases * G);
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(ts.data(), h->phase_ts, ts.size() * sizeof(long long), cudaMemcpyDeviceToHost) !=
          cudaSuccess)
    return MOE_ECUDA;
  for (int p = 0; p + 1 < kPhases; ++p) {
    double sum = 0.0, mx = 0.0;
    for (int l = 0; l < L; ++l) {
      double lmax = 0.0;
      for (int c = 0; c < G; ++c) {
        const double d = (double)(ts[((size_t)l * kPhases + p + 1) * G + c] -
                                  ts[((size_t)l * kPhases + p) * G + c]) * 1e-3;
        sum += d;
        if (d > lmax) lmax = d;
      }
      mx += lmax;
    }
    mean_us[p] = sum / ((double)L * G);
    max_us[p] = mx / L;
  }
  return MOE_OK;
}

}  // extern "C"
