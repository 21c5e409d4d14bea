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
#include <mutex>
#include <vector>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int NT = 256;  // threads per CTA
constexpr int NW = NT / 32;
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
// device waits count SM cycles: 2 cycles per requested ns bounds the wall time between
// ns (at ~2 GHz) and a few times ns at lower clocks
constexpr long long kCyclesPerNs = 2;
constexpr long long kDefaultWaitCycles = (long long)kDefaultWaitNs * kCyclesPerNs;
constexpr int kPhases = 9;  // phase stamps per layer when profiling (8 intervals)

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
  unsigned* bar;      // [0] barrier arrivals, [33] abort flag
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

// A 16-byte block is handled as two 64-bit word pairs D0 = {w0, w1}, D1 = {w2, w3} (and
// the same shifted right by 12 in each half).  ANDing a pair with a slot mask isolates
// slot m of two words at once -- elements (m, 8+m) of D0 and (16+m, 24+m) of D1 -- as
// two subnormal floats already laid out as an f32x2 operand.  Activations are kept as
// matching pairs: xp[m] = (x'[m], x'[8+m]) and xp[8+m] = (x'[16+m], x'[24+m]).
struct BlockPairs {
  f2_t d0, d1, t0, t1;
};

__device__ __forceinline__ BlockPairs block_pairs(const uint4 nb) {
  BlockPairs b;
  asm("mov.b64 %0, {%1,%2};" : "=l"(b.d0) : "r"(nb.x), "r"(nb.y));
  asm("mov.b64 %0, {%1,%2};" : "=l"(b.d1) : "r"(nb.z), "r"(nb.w));
  asm("mov.b64 %0, {%1,%2};" : "=l"(b.t0) : "r"(nb.x >> 12), "r"(nb.y >> 12));
  asm("mov.b64 %0, {%1,%2};" : "=l"(b.t1) : "r"(nb.z >> 12), "r"(nb.w >> 12));
  return b;
}

// slot m's mask in both halves; slots 5..7 are read from the shifted pair
__device__ __forceinline__ f2_t slot_pair(const BlockPairs& b, int half, int m) {
  constexpr f2_t M[5] = {0x0000000F0000000Full, 0x000000F0000000F0ull, 0x00000F0000000F00ull,
                         0x0000F0000000F000ull, 0x000F0000000F0000ull};
  const f2_t d = half ? b.d1 : b.d0;
  const f2_t t = half ? b.t1 : b.t0;
  return (m <= 4) ? (d & M[m]) : (t & M[m - 3]);
}

// Pre-scaled activation pairs of one 32-element block from 32 floats v[k]:
// xp[8h + m] = (v[16h + m] * scale(m), v[16h + 8 + m] * scale(m)).
__device__ __forceinline__ void make_pairs(const float* v, f2_t* xp) {
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int m = 0; m < 8; ++m)
      xp[8 * h + m] = f2pack(v[16 * h + m] * slot_scale(m), v[16 * h + 8 + m] * slot_scale(m));
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

// Each CTA's thread 0 adds 1 to one counter with release semantics (ordering the CTA's
// earlier writes, published to it by the CTA barrier) and polls the counter with
// acquire loads until every CTA of this epoch has arrived.  On this GPU that costs
// about 1.2-1.4 us across both dies; a separate release flag, flag arrays, split
// counters and cluster-first hierarchies all measured slower.  Returns false if the
// round must be abandoned.
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ bool grid_sync(const RoundArgs& a, Sync& sy) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    sy.epoch += 1;
    const unsigned target = sy.epoch * gridDim.x;
    unsigned* abort_flag = a.bar + 33;
    red_release_add(a.bar, 1u);
    int ok = 1;
    const long long t0 = clock64();
    while (ld_acquire(a.bar) < target) {
      if (ld_relaxed(abort_flag)) {
        ok = 0;
        break;
      }
      if (clock64() - t0 > a.wait_cycles) {
        atomicOr(a.status, kStatusTimeout);
        atomicExch(abort_flag, 1u);
        ok = 0;
        break;
      }
    }
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

// Router rows owned by this CTA: experts e = CTA + grid * q (q = 0, 1, ...).  They are
// staged into shared memory by one bulk copy per row, issued as soon as the previous
// layer's expert stream is done (router weights do not depend on any data).
__device__ __forceinline__ int router_rows_of_cta(int E) {
  return (E - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
}

__device__ void issue_router_rows(const RoundArgs& a, const float* router, float* s_rw,
                                  uint32_t bar) {
  const int n = router_rows_of_cta(a.E);
  if (n <= 0) return;
  const uint32_t row_bytes = (uint32_t)a.H * 4u;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(bar, row_bytes * (uint32_t)n);
  for (int q = 0; q < n; ++q) {
    const int e = blockIdx.x + gridDim.x * q;
    bulk_g2s(smem_u32(s_rw + (size_t)q * a.H), router + (size_t)e * a.H, row_bytes, bar);
  }
}

// Lane l accumulates elements 128c + 4l + j for c ascending, then the xor-butterfly.
// Warp q of the CTA computes its staged row q for every activation row.
__device__ void router_phase(const RoundArgs& a, const uint16_t* x, const float* s_rw) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int NC = a.H >> 7;  // <= 16
  const int n = router_rows_of_cta(a.E);
  for (int q = warp; q < n; q += NW) {
    const int e = blockIdx.x + gridDim.x * q;
    const float4* wr = reinterpret_cast<const float4*>(s_rw + (size_t)q * a.H) + lane;
    for (int r = 0; r < a.R; ++r) {
      const uint2* xr = reinterpret_cast<const uint2*>(x + (size_t)r * a.H) + lane;
      uint2 xv[16];
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c < NC) xv[c] = __ldg(xr + 32 * c);
      float p = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        if (c < NC) {
          const float4 w = wr[32 * c];
          p = __fmaf_rn(w.x, bf16_lo(xv[c].x), p);
          p = __fmaf_rn(w.y, bf16_hi(xv[c].x), p);
          p = __fmaf_rn(w.z, bf16_lo(xv[c].y), p);
          p = __fmaf_rn(w.w, bf16_hi(xv[c].y), p);
        }
      }
      p = warp_sum(p);
      if (lane == 0) a.logits[(size_t)r * a.E + e] = p;
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

// True if (ka, ia) ranks before (kb, ib): larger key, then lower id.
__device__ __forceinline__ bool ranks_before(unsigned ka, int ia, unsigned kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// Top-k of one row of logits by one warp.  Lane l owns experts l + 32t (t < NE), kept
// sorted best-first in registers (bitonic network); each of the k rounds takes the
// warp-wide best head (redux.sync max on the key, then min on the id among equal
// keys) and the owning lane pops it.  Lane j returns pick j (logit and id).
template <int NE>
__device__ __forceinline__ void select_row(const float* row, int E, int k, int lane, float& my_l,
                                           int& my_id) {
  unsigned kk[NE];
  int id[NE];
#pragma unroll
  for (int t = 0; t < NE; ++t) {
    const int e = lane + 32 * t;
    id[t] = e;
    kk[t] = (e < E) ? order_key(__ldcg(row + e)) : 0u;
  }
#pragma unroll
  for (int size = 2; size <= NE; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < NE; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;  // this block sorts best-first
          const bool sw = up ? ranks_before(kk[j], id[j], kk[i], id[i])
                             : ranks_before(kk[i], id[i], kk[j], id[j]);
          if (sw) {
            const unsigned tk = kk[i];
            kk[i] = kk[j];
            kk[j] = tk;
            const int ti = id[i];
            id[i] = id[j];
            id[j] = ti;
          }
        }
      }
    }
  }
  for (int j = 0; j < k; ++j) {
    const unsigned m = __reduce_max_sync(0xffffffffu, kk[0]);
    const unsigned cand = (kk[0] == m) ? (unsigned)id[0] : 0xffffffffu;
    const unsigned win = __reduce_min_sync(0xffffffffu, cand);
    if ((unsigned)id[0] == win) {
#pragma unroll
      for (int t = 0; t + 1 < NE; ++t) {
        kk[t] = kk[t + 1];
        id[t] = id[t + 1];
      }
      kk[NE - 1] = 0u;
      id[NE - 1] = INT_MAX;
    }
    if (lane == j) {
      my_l = key_value(m);
      my_id = (int)win;
    }
  }
}

// scratch (inside the staging area, free while routing): mask [E], off_e [E], ids [R*k]
__device__ int route_phase(const RoundArgs& a, const Tables& T, unsigned* s_mask, int* s_off_e,
                           int* s_ids, int layer) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, k = a.k, R = a.R;
  for (int e = tid; e < E; e += NT) s_mask[e] = 0u;
  for (int r = warp; r < R; r += NW) {
    float my_l = 0.f;
    int my_id = 0;
    if (E <= 128)
      select_row<4>(a.logits + (size_t)r * E, E, k, lane, my_l, my_id);
    else  // E <= 512 (moe_create rejects more)
      select_row<16>(a.logits + (size_t)r * E, E, k, lane, my_l, my_id);
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
// Activation pairs of one 32-element block of one row (see make_pairs), built from
// the row's bf16 values, plus -8 * (sum of the block's 32 values).
struct XBlock {
  f2_t xp[16];
  float xsum8;
};

__device__ __forceinline__ void load_xblock(const uint16_t* x, int H, int row, int blk, XBlock& xb) {
  // elements 16h + m and 16h + 8 + m come from 16-byte loads 2h and 2h + 1
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)row * H + 32 * blk);
  float sum = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 ua = __ldg(src + 2 * h), ub = __ldg(src + 2 * h + 1);
    const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float va = (m & 1) ? bf16_hi(wa[m >> 1]) : bf16_lo(wa[m >> 1]);
      const float vb = (m & 1) ? bf16_hi(wb[m >> 1]) : bf16_lo(wb[m >> 1]);
      xb.xp[8 * h + m] = f2pack(va * slot_scale(m), vb * slot_scale(m));
      sum = __fadd_rn(sum, va);
      sum = __fadd_rn(sum, vb);
    }
  }
  xb.xsum8 = -8.f * sum;
}

// Gate/up mapping: lane = one 32-element block; a weight row of H/32 blocks is covered
// by NBL warps (warp w takes blocks 32 * (w % NBL) + lane); the NW / NBL warp groups
// split the 64 weight rows (32 gate, 32 up) of the slice.  Each warp's partial of a row
// goes to s_part[row][w % NBL] and the NBL partials are added in order afterwards.
template <int NBL>
struct GateUpMap {
  static constexpr int kGroups = NW / NBL;     // warp groups
  static constexpr int kRows = 64 / kGroups;   // weight rows per warp
};

// Computes a group of G rows (pairs pp0..pp0+G-1 of the item's expert) against the
// staged item: gate/up for the 64 weight rows, SwiGLU, then the down partials.  Every
// extracted weight pair feeds the G rows, so the integer work is shared.  xb[g] holds
// the lane's activation block of row g.  Waits for the stage's down copies (barrier B)
// before the first down pass if `need_b`.  Ends with a CTA barrier; false on timeout.
template <int NBL, int G>
__device__ __forceinline__ bool compute_group(const RoundArgs& a, const Tables& T, const Stage& st,
                                              int pp0, int s, const XBlock (&xb)[G], float* s_part,
                                              float* s_h, bool& need_b, uint32_t parity_b) {
  const int H = a.H, NB = H >> 5, NS = a.I >> 5;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint8_t* s_gu = st.base;
  const uint16_t* s_gus = reinterpret_cast<const uint16_t*>(st.base + 32 * (size_t)H);
  const uint8_t* s_dn = st.base + 36 * (size_t)H;
  const uint16_t* s_dns = reinterpret_cast<const uint16_t*>(st.base + 52 * (size_t)H);
  using Map = GateUpMap<NBL>;
  const int half = warp % NBL, grp = warp / NBL;
  const int blk = 32 * half + lane;
  // ---- gate / up ----
  float part[Map::kRows][G];
#pragma unroll
  for (int q = 0; q < Map::kRows; ++q)
#pragma unroll
    for (int g = 0; g < G; ++g) part[q][g] = 0.f;
  if (blk < NB) {
#pragma unroll
    for (int q = 0; q < Map::kRows; ++q) {
      const int wr = grp + Map::kGroups * q;
      const uint4 nb = *reinterpret_cast<const uint4*>(s_gu + ((size_t)wr * NB + blk) * 16);
      const float sc = half_bits(s_gus[wr * NB + blk]);
      const BlockPairs bp = block_pairs(nb);
      f2_t acc0[G], acc1[G];
#pragma unroll
      for (int g = 0; g < G; ++g) acc0[g] = acc1[g] = 0ull;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const f2_t e0 = slot_pair(bp, 0, m), e1 = slot_pair(bp, 1, m);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          ffma2(acc0[g], e0, xb[g].xp[m]);
          ffma2(acc1[g], e1, xb[g].xp[8 + m]);
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float dot = __fadd_rn(f2sum(acc0[g]), f2sum(acc1[g]));
        part[q][g] = __fmaf_rn(sc, __fmaf_rn(dot, 0x1p62f, xb[g].xsum8), part[q][g]);
      }
    }
  }
#pragma unroll
  for (int q = 0; q < Map::kRows; ++q)
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float v = warp_sum(part[q][g]);
      if (lane == 0) s_part[((grp + Map::kGroups * q) * 2 + g) * NBL + half] = v;
    }
  __syncthreads();
  // ---- SwiGLU on the slice's 32 intermediate rows, warp g for row g; the scaled h
  // pairs for the down pass go to s_h in pair order (see make_pairs) ----
  if (warp < G) {
    float gg = 0.f, vv = 0.f;
#pragma unroll
    for (int hf = 0; hf < NBL; ++hf) {
      gg = __fadd_rn(gg, s_part[(lane * 2 + warp) * NBL + hf]);
      vv = __fadd_rn(vv, s_part[((32 + lane) * 2 + warp) * NBL + hf]);
    }
    const float hh = __fmul_rn(__fdiv_rn(gg, __fadd_rn(1.f, expf(-gg))), vv);
    // element k = lane: pair index 8 * (k / 16) + (k % 8), component (k / 8) % 2
    float* hrow = s_h + warp * 36;
    hrow[2 * (8 * (lane >> 4) + (lane & 7)) + ((lane >> 3) & 1)] = hh * slot_scale(lane & 7);
    const float hs = warp_sum(hh);
    if (lane == 0) hrow[32] = -8.f * hs;
  }
  if (need_b) {
    const bool ok = mbar_wait_bounded(st.bar_b, parity_b, a.status, a.wait_cycles);
    if (__syncthreads_or(!ok)) return false;
    need_b = false;
  } else {
    __syncthreads();
  }
  // ---- down partials: thread per output row, one 32-element K-block each ----
  f2_t hp[G][16];
  float hsum8[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const f2_t* hrow = reinterpret_cast<const f2_t*>(s_h + g * 36);
#pragma unroll
    for (int q = 0; q < 16; ++q) hp[g][q] = hrow[q];
    hsum8[g] = s_h[g * 36 + 32];
  }
  int pair[G];
#pragma unroll
  for (int g = 0; g < G; ++g) pair[g] = T.pair[pp0 + g];
  for (int o = tid; o < H; o += NT) {
    const uint4 nb = *reinterpret_cast<const uint4*>(s_dn + (size_t)o * 16);
    const float sc = half_bits(s_dns[o]);
    const BlockPairs bp = block_pairs(nb);
    f2_t acc0[G], acc1[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc0[g] = acc1[g] = 0ull;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const f2_t e0 = slot_pair(bp, 0, m), e1 = slot_pair(bp, 1, m);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        ffma2(acc0[g], e0, hp[g][m]);
        ffma2(acc1[g], e1, hp[g][8 + m]);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float dot = __fadd_rn(f2sum(acc0[g]), f2sum(acc1[g]));
      a.partial[((size_t)pair[g] * NS + s) * H + o] = __fmul_rn(sc, __fmaf_rn(dot, 0x1p62f, hsum8[g]));
    }
  }
  // the next group's gate/up may overwrite s_part / s_h only after everyone is done here
  __syncthreads();
  return true;
}

// Stage b's state lives in two bitfields: `ph` holds the parity to wait for (bit 2b:
// gate/up barrier A, bit 2b+1: down barrier B) and `pend` marks copies in flight.  On
// success both barriers have been consumed (parities flipped, pending bits cleared);
// on failure `pend` still marks the copies the caller must drain.
template <int NBL>
__device__ __forceinline__ bool compute_item(const RoundArgs& a, const Tables& T, const Stage& st, int b,
                             unsigned& ph, unsigned& pend, int ui, int s, const uint16_t* x,
                             float* s_part, float* s_h, int stamp_layer) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int blk = 32 * (warp % NBL) + lane;
  const bool has_blk = blk < (a.H >> 5);
  const unsigned bit_a = 1u << (2 * b), bit_b = 2u << (2 * b);
  bool ok = mbar_wait_bounded(st.bar_a, (ph & bit_a) ? 1u : 0u, a.status, a.wait_cycles);
  if (__syncthreads_or(!ok)) return false;
  ph ^= bit_a;
  pend &= ~bit_a;
  if (stamp_layer >= 0) stamp(a, stamp_layer, 4);
  bool need_b = true;
  const uint32_t parity_b = (ph & bit_b) ? 1u : 0u;
  const int p0 = T.csr_off[ui], p1 = T.csr_off[ui + 1];
  int pp = p0;
  for (; pp + 2 <= p1; pp += 2) {
    XBlock xb2[2];
    if (has_blk) {
      load_xblock(x, a.H, T.pair[pp] / a.k, blk, xb2[0]);
      load_xblock(x, a.H, T.pair[pp + 1] / a.k, blk, xb2[1]);
    }
    if (!compute_group<NBL, 2>(a, T, st, pp, s, xb2, s_part, s_h, need_b, parity_b)) return false;
  }
  if (pp < p1) {
    XBlock xb1[1];
    if (has_blk) load_xblock(x, a.H, T.pair[pp] / a.k, blk, xb1[0]);
    if (!compute_group<NBL, 1>(a, T, st, pp, s, xb1, s_part, s_h, need_b, parity_b)) return false;
  }
  if (need_b) {  // (every union expert has a row, so this only keeps phases paired)
    ok = mbar_wait_bounded(st.bar_b, parity_b, a.status, a.wait_cycles);
    if (__syncthreads_or(!ok)) return false;
  }
  ph ^= bit_b;
  pend &= ~bit_b;
  return true;
}

// ---------------------------------------------------------------------------------
// P4: fixed-order weighted reduction of the partials into the layer output

// Tile = (row r, 32 consecutive outputs).  Unit u = (rank j, part): a warp sums the
// partials of slices s = part, part + jw, ... for its 32 outputs (coalesced), then warp
// 0 combines: y_j = sum over parts in order, out = sum_j w_j y_j in rank order.
__device__ void reduce_phase(const RoundArgs& a, const Tables& T, float* out, float* s_red) {
  const int H = a.H, k = a.k, NS = a.I >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int jw = (NW / k) > 0 ? (NW / k) : 1;  // warps per rank
  const int units = k * jw;
  const int tiles_per_row = H >> 5;
  const int n_tiles = a.R * tiles_per_row;
  for (int q = blockIdx.x; q < n_tiles; q += gridDim.x) {
    const int r = q / tiles_per_row;
    const int o0 = (q - r * tiles_per_row) * 32;
    for (int u = warp; u < units; u += NW) {
      const int j = u / jw, part = u - (u / jw) * jw;
      const float* src = a.partial + (size_t)(r * k + j) * NS * H + o0 + lane;
      float y = 0.f;
#pragma unroll 8
      for (int s = part; s < NS; s += jw) y = __fadd_rn(y, __ldcg(src + (size_t)s * H));
      s_red[u * 32 + lane] = y;
    }
    __syncthreads();
    if (warp == 0) {
      float acc = 0.f;
      for (int j = 0; j < k; ++j) {
        float yj = 0.f;
        for (int part = 0; part < jw; ++part) yj = __fadd_rn(yj, s_red[(j * jw + part) * 32 + lane]);
        acc = __fmaf_rn(T.w[r * k + j], yj, acc);
      }
      out[(size_t)r * H + o0 + lane] = acc;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------------
// shared-memory plan

constexpr size_t kRouterOffset = 8192;  // reduction scratch (<= 4 KB) sits below

struct SmemPlan {
  size_t stage, stage0, stage1, router, bars, gv, uni, csr, pair, w, nunion, total;
  bool router_fits;
};

__host__ __device__ inline size_t up128(size_t x) { return (x + 127) & ~(size_t)127; }

// router_rows = experts per CTA, ceil(E / grid)
__host__ __device__ inline SmemPlan smem_plan(int H, int E, int R, int k, int router_rows) {
  SmemPlan p{};
  p.stage = up128(stage_bytes(H));
  size_t off = 0;
  p.stage0 = off;  off += p.stage;
  p.stage1 = off;  off += p.stage;
  // The next layer's router rows live in stage 1 after the reduction scratch: they are
  // written after the last expert item of a layer and read before the next layer's
  // first item, while the staging buffers are idle.
  p.router = p.stage1 + kRouterOffset;
  p.router_fits = kRouterOffset + (size_t)router_rows * H * 4 <= p.stage;
  p.bars = off;    off += 64;
  p.gv = off;      off += up128((256 + 72) * 4);
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
  const SmemPlan P = smem_plan(a.H, a.E, a.R, a.k, (a.E + (int)gridDim.x - 1) / (int)gridDim.x);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bars);
  const uint32_t bar_router = smem_u32(bars + 4);
  float* s_rw = reinterpret_cast<float*>(smem + P.router);
  // stage b: buffer at stage0 + b * stage, barriers bars[2b] (A) and bars[2b + 1] (B)
  auto stage_of = [&](int b) {
    return Stage{smem + P.stage0 + (size_t)b * P.stage, smem_u32(bars + 2 * b),
                 smem_u32(bars + 2 * b + 1)};
  };
  float* s_part = reinterpret_cast<float*>(smem + P.gv);  // [64 weight rows][2 group rows][NBL]
  float* s_h = s_part + 256;                               // [2][36]: 16 h pairs + -8 sum(h)
  Tables T{reinterpret_cast<int*>(smem + P.uni), reinterpret_cast<int*>(smem + P.csr),
           reinterpret_cast<int*>(smem + P.pair), reinterpret_cast<float*>(smem + P.w),
           reinterpret_cast<int*>(smem + P.nunion)};
  // routing scratch lives in the (then idle) staging area
  unsigned* s_mask = reinterpret_cast<unsigned*>(smem + P.stage0);
  int* s_off_e = reinterpret_cast<int*>(smem + P.stage0 + (size_t)a.E * 4);
  int* s_ids = reinterpret_cast<int*>(smem + P.stage0 + (size_t)a.E * 8);
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(smem_u32(bars + i), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    issue_router_rows(a, a.layer[0].router, s_rw, bar_router);
  }
  __syncthreads();
  unsigned ph_router = 0u;
  bool router_pend = router_rows_of_cta(a.E) > 0;  // layer 0's rows are in flight

  Sync sy;
  unsigned ph = 0u;    // parity to wait for: bit 2b = stage b's barrier A, bit 2b+1 = B
  unsigned pend = 0u;  // copies in flight, same bit layout
  // Leaving early: give every copy still in flight a bounded chance to land (so no
  // bulk copy targets shared memory of an exited CTA), raise the abort flag, return.
  auto bail = [&]() {
    for (int q = 0; q < 4; ++q)
      if (pend & (1u << q))
        mbar_wait_bounded(smem_u32(bars + q), (ph >> q) & 1u, a.status, kDefaultWaitCycles);
    if (router_pend) mbar_wait_bounded(bar_router, ph_router, a.status, kDefaultWaitCycles);
    if (tid == 0) atomicExch(a.bar + 33, 1u);
  };
  const int G = gridDim.x, NS = a.I >> 5;
  const size_t RH = (size_t)a.R * a.H;
  for (int l = 0; l < a.L; ++l) {
    const LayerPtrs& W = a.layer[l];
    const uint16_t* x = a.x + (size_t)l * RH;
    stamp(a, l, 0);
    if (router_pend) {
      const bool ok = mbar_wait_bounded(bar_router, ph_router, a.status, a.wait_cycles);
      if (__syncthreads_or(!ok)) {
        bail();
        return;
      }
      ph_router ^= 1u;
      router_pend = false;
    }
    router_phase(a, x, s_rw);
    stamp(a, l, 1);
    if (!grid_sync(a, sy)) {  // B1: all logits written
      bail();
      return;
    }
    stamp(a, l, 2);
    const int U = route_phase(a, T, s_mask, s_off_e, s_ids, l);
    stamp(a, l, 3);
    if (a.route_only) return;
    const int n_items = U * NS;
    if (blockIdx.x >= n_items) stamp(a, l, 4);  // no item: "first data" = now
    for (int n = 0; n < 2; ++n) {
      const int it = blockIdx.x + n * G;
      if (it < n_items) {
        pend |= 3u << (2 * n);  // every thread tracks what thread 0 issues
        if (tid == 0) issue_item(a, W, stage_of(n), T.uni[it / NS], it % NS);
      }
    }
    for (int n = 0;; ++n) {
      const int it = blockIdx.x + n * G;
      if (it >= n_items) break;
      const int b = n & 1;
      if (!compute_item<NBL>(a, T, stage_of(b), b, ph, pend, it / NS, it % NS, x, s_part, s_h,
                             n == 0 ? l : -1)) {
        bail();
        return;
      }
      // compute_item ends with a CTA barrier: the stage is free again
      const int nxt = it + 2 * G;
      if (nxt < n_items) {
        pend |= 3u << (2 * b);
        if (tid == 0) issue_item(a, W, stage_of(b), T.uni[nxt / NS], nxt % NS);
      }
    }
    // the next layer's router rows can move in now: they do not depend on any data
    if (l + 1 < a.L && router_rows_of_cta(a.E) > 0) {
      router_pend = true;
      if (tid == 0) issue_router_rows(a, a.layer[l + 1].router, s_rw, bar_router);
    }
    stamp(a, l, 5);
    if (!grid_sync(a, sy)) {  // B2: all partials written
      bail();
      return;
    }
    stamp(a, l, 6);
    reduce_phase(a, T, a.out + (size_t)l * RH, reinterpret_cast<float*>(smem + P.stage1));
    stamp(a, l, 7);
    if (l + 1 < a.L && !grid_sync(a, sy)) {  // B3: layer output complete
      bail();
      return;
    }
    stamp(a, l, 8);  // (the last layer has no B3: its interval is zero)
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

size_t smem_bytes(const moe_dims& d, int rows, int grid) {
  return smem_plan(d.hidden, d.n_experts, rows, d.top_k, (d.n_experts + grid - 1) / grid).total;
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
  cfg.dynamicSmemBytes = smem_bytes(h->dims, a.R, h->sm_count);
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
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  DeviceGuard g(device);
  if (!g.ok) return MOE_ECUDA;
  int coop = 0, sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device) != cudaSuccess || !coop) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  const size_t smem = smem_bytes(*dims, dims->max_rows, sms);
  const SmemPlan plan = smem_plan(dims->hidden, dims->n_experts, dims->max_rows, dims->top_k,
                                  (dims->n_experts + sms - 1) / sms);
  if (smem + 1024 > 227 * 1024 || !plan.router_fits) return MOE_EUNSUPPORTED;
  moe_handle* h = new moe_handle();
  h->dims = *dims;
  h->device = device;
  h->sm_count = sms;
  if (cudaMalloc(&h->status, sizeof(unsigned)) != cudaSuccess ||
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

// =====================================================================================
// Allocation-free variant of moe_decode_layer.
//
// Some callers cannot allocate device memory at all: code that runs inside another
// framework's memory pool with allocation disabled, allocation-free real-time or
// embedded loops, or hosts that forbid cudaMalloc after start-up.  For them the
// workspace (grid-barrier words, router logits, split-K partials) lives in the file-
// scope array below, which the CUDA runtime places on every device that loads this
// library and keeps until the process exits.  The caller passes only inputs and
// outputs; this path calls no cudaMalloc, cudaFree or allocating library routine.

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;  // 16 MiB per device
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
  bool ready = false;
  void* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int sms = 0;
};

NoAllocDevice g_noalloc[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

// One-time set-up of the current device: the device address of the scratch array (in
// host code the symbol names a host-side stand-in, not device memory), the SM count,
// and the kernel's shared-memory attribute.
int noalloc_setup(int dev, size_t smem, NoAllocDevice** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return MOE_ECUDA;
    }
    int sms = 0, coop = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) {
      cudaGetLastError();
      return MOE_ECUDA;
    }
    d.scratch = p;
    d.sms = sms;
    d.ready = true;
  }
  cudaError_t e = cudaFuncSetAttribute(k_round<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_round<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  *out = &d;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_decode_layer_noalloc(const moe_dims* dims, const moe_layer_w* w,
                                        const uint16_t* x_bf16, int32_t rows, float* out,
                                        unsigned* dev_status, void* stream) {
  int rc = check_dims(dims);
  if (rc != MOE_OK) return rc;
  if ((rc = check_layer(w)) != MOE_OK) return rc;
  if (!aligned16(x_bf16) || !aligned16(out) || rows < 1 || rows > dims->max_rows)
    return MOE_EINVAL;
  if (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3u)) return MOE_EINVAL;
  // the scratch holds the status word (first 256 bytes) and the layer's workspace
  const WsLayout L = ws_layout(*dims, rows);
  if (256 + L.total > kNoAllocScratchBytes) return MOE_EWORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  const size_t smem = smem_bytes(*dims, rows, sms);
  const SmemPlan plan = smem_plan(dims->hidden, dims->n_experts, rows, dims->top_k,
                                  (dims->n_experts + sms - 1) / sms);
  if (smem + 1024 > 227 * 1024 || !plan.router_fits) return MOE_EUNSUPPORTED;
  NoAllocDevice* d = nullptr;
  if ((rc = noalloc_setup(dev, smem, &d)) != MOE_OK) return rc;
  char* base = static_cast<char*>(d->scratch);
  unsigned* own_status = reinterpret_cast<unsigned*>(base);
  void* ws = base + 256;
  RoundArgs a{};
  const moe_dims& dd = *dims;
  a.H = dd.hidden;
  a.E = dd.n_experts;
  a.k = dd.top_k;
  a.I = dd.inter;
  a.R = rows;
  a.L = 1;
  a.bar = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + L.ctrl);
  a.logits = reinterpret_cast<float*>(static_cast<char*>(ws) + L.logits);
  a.partial = reinterpret_cast<float*>(static_cast<char*>(ws) + L.partial);
  a.status = dev_status ? dev_status : own_status;
  a.wait_cycles = kDefaultWaitCycles;
  a.x = x_bf16;
  a.out = out;
  copy_layers(a, w, 1);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the barrier words must start at zero; logits and partials are fully overwritten
  if (cudaMemsetAsync(a.bar, 0, 256, st) != cudaSuccess) return MOE_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = (nbl_of(a.H) == 1) ? cudaLaunchKernelEx(&cfg, k_round<1>, a)
                                           : cudaLaunchKernelEx(&cfg, k_round<2>, a);
  return e == cudaSuccess ? MOE_OK : MOE_ECUDA;
}
