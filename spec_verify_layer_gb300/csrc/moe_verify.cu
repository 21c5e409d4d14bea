// GB300 (sm_103a) kernels and C ABI of the MoE layer of a speculative-decoding
// verify round.  See include/moe_verify.h for the operation and the contract.
//
// Per layer, three kernels in stream order:
//   k_route   router GEMV (one warp per expert, canonical fp32 order), then the last
//             CTA to finish selects each row's top-k, the renormalised weights, the
//             ascending expert union and a CSR list of (row, rank) pairs per expert.
//   k_expert  split-K over the expert intermediate dimension: work item = (union
//             expert u, slice of 32 intermediate rows).  One elected thread stages the
//             item's gate/up rows, their scales, the matching down K-block and its
//             scales into shared memory with 1-D bulk TMA copies (one mbarrier); the
//             CTA then computes g, v, h = silu(g) v for its rows and the down partial
//             Wd[:, slice] h[slice], written per (row, rank, slice) to the workspace.
//   k_reduce  out[r][o] = sum_j w[r][j] * sum_s partial[r, j, s][o] in a fixed order,
//             so a row's result depends only on that row (bitwise).
//
// Dequantisation in registers without a convert instruction: a nibble n placed in
// bits [p, p+4) of an otherwise-zero fp32 word is the subnormal n * 2^(p-149), and an
// fma with x * 2^(87-4m) (m = the nibble's slot) yields n * x * 2^-62 exactly.  A
// 32-bit word of 8 nibbles therefore costs one AND per weight (plus one shift for the
// top three nibbles) and one FFMA per weight and row.  The code offset (q = n - 8) is
// applied once per 32-element block: sum (n-8) x = 2^62 acc - 8 sum x.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <vector>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
// device waits count SM cycles: 2 cycles per requested ns bounds the wall time between
// ns (at ~2 GHz) and a few times ns at lower clocks
constexpr long long kCyclesPerNs = 2;
constexpr long long kDefaultWaitCycles = (long long)kDefaultWaitNs * kCyclesPerNs;

struct Ctrl {
  unsigned ticket;   // k_route: CTAs that finished their logits
  unsigned n_union;  // |U| of the current layer
  unsigned pad[62];
};

struct LayerArgs {
  int H, E, k, I, R;
  const float* router;
  const uint8_t* gu_nib;
  const uint16_t* gu_sc;
  const uint8_t* dn_nib;
  const uint16_t* dn_sc;
  const uint16_t* x;  // [R][H] bf16 bits
  float* out;         // [R][H]
  // workspace
  Ctrl* ctrl;
  float* logits;   // [R][E]
  int* ids;        // [R][k]
  float* w;        // [R][k]
  int* uni;        // [E]
  int* csr_off;    // [E+1]
  int* csr_pair;   // [R*k]
  float* partial;  // [R*k][I/32][H]
  // optional caller outputs of moe_route, and the per-layer |U| slot of moe_round
  int* user_ids;
  float* user_w;
  int* user_union;
  int* user_nunion;
  int* stats_slot;
  unsigned* status;
  long long wait_cycles;
};

// ---------------------------------------------------------------------------------
// small device helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
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

// Waits for `phase` of the mbarrier for at most `limit` SM clock cycles; on giving up
// it raises the timeout bit of the status word and returns false.  The first poll
// does not block, so a bound of a few cycles gives up deterministically.
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

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// 2^(87 - 4m) for nibble slots m = 0..4 and 2^(99 - 4m) for m = 5..7 (those three are
// read after a 12-bit right shift): the factor that turns the subnormal n * 2^e_m into
// n * x * 2^-62 under an fma.
__device__ __forceinline__ float slot_scale(int m) {
  const int e = (m <= 4) ? 87 - 4 * m : 99 - 4 * m;
  return __int_as_float((127 + e) << 23);
}

// acc += sum over the 8 nibbles of w of n_m * xs[m] (xs pre-scaled by slot_scale).
__device__ __forceinline__ void dot8(uint32_t w, const float* xs, float& acc) {
  acc = __fmaf_rn(__uint_as_float(w & 0x0000000Fu), xs[0], acc);
  acc = __fmaf_rn(__uint_as_float(w & 0x000000F0u), xs[1], acc);
  acc = __fmaf_rn(__uint_as_float(w & 0x00000F00u), xs[2], acc);
  acc = __fmaf_rn(__uint_as_float(w & 0x0000F000u), xs[3], acc);
  acc = __fmaf_rn(__uint_as_float(w & 0x000F0000u), xs[4], acc);
  const uint32_t t = w >> 12;
  acc = __fmaf_rn(__uint_as_float(t & 0x00000F00u), xs[5], acc);
  acc = __fmaf_rn(__uint_as_float(t & 0x0000F000u), xs[6], acc);
  acc = __fmaf_rn(__uint_as_float(t & 0x000F0000u), xs[7], acc);
}

// 2^-62 * sum_{k<32} n_k x_k for one 16-byte block of codes.
__device__ __forceinline__ float dot32(const uint4 nb, const float* xs) {
  float a0 = 0.f, a1 = 0.f;
  dot8(nb.x, xs + 0, a0);
  dot8(nb.y, xs + 8, a1);
  dot8(nb.z, xs + 16, a0);
  dot8(nb.w, xs + 24, a1);
  return __fadd_rn(a0, a1);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ float half_bits(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// ---------------------------------------------------------------------------------
// step 1: router logits, one warp per expert, canonical order

__device__ void router_logits_warp(const LayerArgs& a, int e, int lane) {
  const int NC = a.H >> 7;  // <= 16
  const float4* wr = reinterpret_cast<const float4*>(a.router + (size_t)e * a.H) + lane;
  float4 wv[16];
#pragma unroll
  for (int c = 0; c < 16; ++c)
    if (c < NC) wv[c] = __ldg(wr + 32 * c);
  for (int r = 0; r < a.R; ++r) {
    const uint2* xr = reinterpret_cast<const uint2*>(a.x + (size_t)r * a.H) + lane;
    float p = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      if (c < NC) {
        const uint2 xv = __ldg(xr + 32 * c);
        p = __fmaf_rn(wv[c].x, bf16_lo(xv.x), p);
        p = __fmaf_rn(wv[c].y, bf16_hi(xv.x), p);
        p = __fmaf_rn(wv[c].z, bf16_lo(xv.y), p);
        p = __fmaf_rn(wv[c].w, bf16_hi(xv.y), p);
      }
    }
    p = warp_sum(p);
    if (lane == 0) a.logits[(size_t)r * a.E + e] = p;
  }
}

// ---------------------------------------------------------------------------------
// steps 2-3: per-row top-k + weights, union, CSR -- executed by one CTA

__device__ void topk_union_cta(const LayerArgs& a) {
  __shared__ int s_ids[kMaxRows * kMaxTopK];
  __shared__ unsigned s_mask[kMaxExperts];  // rows that picked expert e
  __shared__ int s_off[kMaxExperts];        // CSR offset of e
  __shared__ int s_wf[NW], s_wc[NW];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, k = a.k, R = a.R;
  for (int e = tid; e < E; e += NT) s_mask[e] = 0u;

  const int NE = (E + 31) >> 5;  // <= 32
  for (int r = warp; r < R; r += NW) {
    float v[32];
    unsigned taken = 0u;
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      if (t < NE) {
        const int e = lane + 32 * t;
        if (e < E) {
          v[t] = __ldcg(a.logits + (size_t)r * E + e);
        } else {
          v[t] = -INFINITY;
          taken |= 1u << t;
        }
      }
    }
    float my_l = 0.f;
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = INT_MAX;
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        if (t < NE && !((taken >> t) & 1u)) {
          const int e = lane + 32 * t;
          if (ranks_before(v[t], e, bv, bi)) {
            bv = v[t];
            bi = e;
          }
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ranks_before(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == j) {
        my_l = bv;
        my_id = bi;
      }
    }
    // renormalised weights: exp(l_j - l_1) / sum over the k picks, summed in rank order
    const float l1 = __shfl_sync(0xffffffffu, my_l, 0);
    const float ex = (lane < k) ? expf(my_l - l1) : 0.f;
    float den = 0.f;
    for (int j = 0; j < k; ++j) den = __fadd_rn(den, __shfl_sync(0xffffffffu, ex, j));
    if (lane < k) {
      const float wj = __fdiv_rn(ex, den);
      const int p = r * k + lane;
      s_ids[p] = my_id;
      a.ids[p] = my_id;
      a.w[p] = wj;
      if (a.user_ids) a.user_ids[p] = my_id;
      if (a.user_w) a.user_w[p] = wj;
    }
  }
  __syncthreads();
  for (int p = tid; p < R * k; p += NT) atomicOr(&s_mask[s_ids[p]], 1u << (p / k));
  __syncthreads();

  // exclusive scans over e of (picked ? 1 : 0) and popc(mask): union index, CSR offset
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
      s_off[e] = basec;
      a.uni[basef] = e;
      a.csr_off[basef] = basec;
      if (a.user_union) a.user_union[basef] = e;
      ++basef;
      basec += __popc(m);
    }
  }
  if (tid == NT - 1) {
    // the last thread's inclusive totals are the union size and the pair count
    a.ctrl->n_union = (unsigned)basef;
    a.csr_off[basef] = basec;
    if (a.user_nunion) *a.user_nunion = basef;
    if (a.stats_slot) *a.stats_slot = basef;
  }
  __syncthreads();
  for (int p = tid; p < R * k; p += NT) {
    const int e = s_ids[p], r = p / k;
    const int pos = s_off[e] + __popc(s_mask[e] & ((1u << r) - 1u));
    a.csr_pair[pos] = p;
  }
}

__global__ void __launch_bounds__(NT) k_route(LayerArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * NW + warp;
  if (e < a.E) router_logits_warp(a, e, lane);
  __threadfence();
  __syncthreads();
  __shared__ unsigned s_last;
  if (threadIdx.x == 0) s_last = (atomicAdd(&a.ctrl->ticket, 1u) == gridDim.x - 1) ? 1u : 0u;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  topk_union_cta(a);
  if (threadIdx.x == 0) a.ctrl->ticket = 0u;
}

// ---------------------------------------------------------------------------------
// steps 4-5a: expert work items

// Shared-memory layout of one staged item (H = hidden):
//   [0, 32H)    gate/up codes: 2 x 32 rows x H/32 blocks x 16 B
//   [32H, 36H)  gate/up scales (fp16)
//   [36H, 52H)  down codes of the slice: H rows x 16 B
//   [52H, 54H)  down scales (fp16)
//   then gv[64] floats, h'[32] floats, hsum, mbarrier
__host__ __device__ constexpr size_t stage_bytes(int H) { return (size_t)54 * H; }
__host__ __device__ constexpr size_t expert_smem_bytes(int H) {
  return stage_bytes(H) + 64 * 4 + 32 * 4 + 16 + 16;
}

template <int NBL>  // blocks of 32 per lane per weight row: ceil(H / 1024)
__global__ void __launch_bounds__(NT, 2) k_expert(LayerArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int H = a.H, NB = H >> 5, NS = a.I >> 5;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* s_gu = smem;
  const uint16_t* s_gus = reinterpret_cast<const uint16_t*>(smem + 32 * (size_t)H);
  const uint8_t* s_dn = smem + 36 * (size_t)H;
  const uint16_t* s_dns = reinterpret_cast<const uint16_t*>(smem + 52 * (size_t)H);
  float* s_gv = reinterpret_cast<float*>(smem + stage_bytes(H));
  float* s_h = s_gv + 64;
  float* s_hsum = s_h + 32;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_hsum + 4);
  const uint32_t bar = smem_u32(s_bar);
  if (tid == 0) mbar_init(bar, 1);
  __syncthreads();

  uint32_t phase = 0;
  const int n_items = (int)__ldcg(&a.ctrl->n_union) * NS;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const int ui = it / NS, s = it - (it / NS) * NS;
    const int u = __ldcg(a.uni + ui);
    if (tid == 0) {
      const size_t I = (size_t)a.I, Hs = (size_t)H;
      // order the previous item's shared-memory reads before the async-proxy writes
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_expect_tx(bar, (uint32_t)stage_bytes(H));
      bulk_g2s(smem_u32(s_gu), a.gu_nib + (size_t)u * I * Hs + (size_t)s * 32 * Hs, 32 * H, bar);
      bulk_g2s(smem_u32(s_gus), a.gu_sc + (size_t)u * (I * Hs / 16) + (size_t)s * 64 * NB, 4 * H,
               bar);
      bulk_g2s(smem_u32(s_dn), a.dn_nib + (size_t)u * (I * Hs / 2) + (size_t)s * 16 * Hs, 16 * H,
               bar);
      bulk_g2s(smem_u32(s_dns), a.dn_sc + (size_t)u * (I * Hs / 32) + (size_t)s * Hs, 2 * H, bar);
    }
    const int p0 = __ldcg(a.csr_off + ui), p1 = __ldcg(a.csr_off + ui + 1);
    bool ok = mbar_wait_bounded(bar, phase, a.status, a.wait_cycles);
    if (__syncthreads_or(!ok)) {
      // give the copies in flight a second bounded chance to land, then leave
      mbar_wait_bounded(bar, phase, a.status, kDefaultWaitCycles);
      break;
    }
    phase ^= 1u;

    for (int pp = p0; pp < p1; ++pp) {
      const int pair = __ldcg(a.csr_pair + pp);
      const int r = pair / a.k;
      // ---- gate / up: warp per weight row, lane per 32-element block ----
      float xs[NBL][32];
      float xsum8[NBL];
#pragma unroll
      for (int t = 0; t < NBL; ++t) {
        const int b = lane + 32 * t;
        xsum8[t] = 0.f;
        if (b < NB) {
          const uint4* xp = reinterpret_cast<const uint4*>(a.x + (size_t)r * H + 32 * b);
          float sum = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 v = __ldg(xp + q);
            const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int z = 0; z < 4; ++z) {
              const float lo = bf16_lo(wds[z]), hi = bf16_hi(wds[z]);
              const int k0 = 8 * q + 2 * z;
              xs[t][k0] = lo * slot_scale(k0 & 7);
              xs[t][k0 + 1] = hi * slot_scale((k0 + 1) & 7);
              sum = __fadd_rn(sum, lo);
              sum = __fadd_rn(sum, hi);
            }
          }
          xsum8[t] = -8.f * sum;
        }
      }
      for (int wr = warp; wr < 64; wr += NW) {
        float part = 0.f;
#pragma unroll
        for (int t = 0; t < NBL; ++t) {
          const int b = lane + 32 * t;
          if (b < NB) {
            const uint4 nb = *reinterpret_cast<const uint4*>(s_gu + ((size_t)wr * NB + b) * 16);
            const float sc = half_bits(s_gus[wr * NB + b]);
            const float acc = dot32(nb, xs[t]);
            part = __fmaf_rn(sc, __fmaf_rn(acc, 0x1p62f, xsum8[t]), part);
          }
        }
        part = warp_sum(part);
        if (lane == 0) s_gv[wr] = part;
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
      __syncthreads();
      // ---- down partial: thread per output row, one 32-element K-block each ----
      float hreg[32];
#pragma unroll
      for (int q = 0; q < 32; ++q) hreg[q] = s_h[q];
      const float hsum8 = *s_hsum;
      float* dst = a.partial + ((size_t)pair * NS + s) * H;
      for (int o = tid; o < H; o += NT) {
        const uint4 nb = *reinterpret_cast<const uint4*>(s_dn + (size_t)o * 16);
        const float sc = half_bits(s_dns[o]);
        const float acc = dot32(nb, hreg);
        dst[o] = __fmul_rn(sc, __fmaf_rn(acc, 0x1p62f, hsum8));
      }
      __syncthreads();
    }
  }
}

// ---------------------------------------------------------------------------------
// step 5b: weighted, fixed-order reduction of the partials

__global__ void __launch_bounds__(NT) k_reduce(LayerArgs a) {
  const int o = blockIdx.x * NT + threadIdx.x;
  const int r = blockIdx.y;
  if (o >= a.H) return;
  const int NS = a.I >> 5;
  float acc = 0.f;
  for (int j = 0; j < a.k; ++j) {
    const int pair = r * a.k + j;
    const float* src = a.partial + (size_t)pair * NS * a.H + o;
    float y = 0.f;
    for (int s = 0; s < NS; ++s) y = __fadd_rn(y, __ldcg(src + (size_t)s * a.H));
    acc = __fmaf_rn(__ldcg(a.w + pair), y, acc);
  }
  a.out[(size_t)r * a.H + o] = acc;
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

struct ProfPair {
  cudaEvent_t start = nullptr, stop = nullptr;
  int kind = 0;
};

struct moe_handle {
  moe_dims dims;
  int device = 0;
  int sm_count = 0;
  int expert_ctas_per_sm = 1;
  unsigned* status = nullptr;
  unsigned long long wait_ns = kDefaultWaitNs;
  int32_t last_launches = 0;
  GraphKey gkey;
  cudaGraphExec_t gexec = nullptr;
  int32_t graph_launches = 0;
  // per-kernel event timing of eager launches (moe_profile)
  bool profiling = false;
  std::vector<ProfPair> prof;
  size_t prof_used = 0;
};

namespace {

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
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

LayerArgs make_args(const moe_handle* h, const moe_layer_w* w, const uint16_t* x, int rows,
                    float* out, void* ws) {
  const moe_dims& d = h->dims;
  const WsLayout L = ws_layout(d, rows);
  char* base = static_cast<char*>(ws);
  LayerArgs a{};
  a.H = d.hidden;
  a.E = d.n_experts;
  a.k = d.top_k;
  a.I = d.inter;
  a.R = rows;
  a.router = w->router;
  a.gu_nib = w->gateup_nib;
  a.gu_sc = w->gateup_scale;
  a.dn_nib = w->down_nib;
  a.dn_sc = w->down_scale;
  a.x = x;
  a.out = out;
  a.ctrl = reinterpret_cast<Ctrl*>(base + L.ctrl);
  a.logits = reinterpret_cast<float*>(base + L.logits);
  a.ids = reinterpret_cast<int*>(base + L.ids);
  a.w = reinterpret_cast<float*>(base + L.w);
  a.uni = reinterpret_cast<int*>(base + L.uni);
  a.csr_off = reinterpret_cast<int*>(base + L.csr_off);
  a.csr_pair = reinterpret_cast<int*>(base + L.csr_pair);
  a.partial = reinterpret_cast<float*>(base + L.partial);
  a.status = h->status;
  const unsigned long long ns = h->wait_ns < (1ull << 40) ? h->wait_ns : (1ull << 40);
  a.wait_cycles = (long long)ns * kCyclesPerNs;
  return a;
}

int expert_grid(const moe_handle* h, int rows) {
  const moe_dims& d = h->dims;
  const int max_u = d.n_experts < rows * d.top_k ? d.n_experts : rows * d.top_k;
  const int max_items = max_u * (d.inter / kSlice);
  const int cap = h->sm_count * h->expert_ctas_per_sm;
  return max_items < cap ? max_items : cap;
}

// Event pair around one launch when profiling eager calls; nullptr otherwise.
ProfPair* prof_begin(moe_handle* h, bool capturing, int kind, cudaStream_t st) {
  if (!h->profiling || capturing) return nullptr;
  if (h->prof_used == h->prof.size()) {
    ProfPair p;
    if (cudaEventCreate(&p.start) != cudaSuccess || cudaEventCreate(&p.stop) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    h->prof.push_back(p);
  }
  ProfPair* p = &h->prof[h->prof_used++];
  p->kind = kind;
  cudaEventRecord(p->start, st);
  return p;
}

void prof_end(ProfPair* p, cudaStream_t st) {
  if (p) cudaEventRecord(p->stop, st);
}

// Enqueues one layer: route (+ top-k/union), optionally expert + reduce.
cudaError_t enqueue_layer(moe_handle* h, const LayerArgs& a, bool full, cudaStream_t st,
                          int32_t* launches, bool capturing = false) {
  const int H = a.H;
  ProfPair* p = prof_begin(h, capturing, 0, st);
  k_route<<<(a.E + NW - 1) / NW, NT, 0, st>>>(a);
  prof_end(p, st);
  ++*launches;
  if (full) {
    const int grid = expert_grid(h, a.R);
    const size_t smem = expert_smem_bytes(H);
    p = prof_begin(h, capturing, 1, st);
    if (nbl_of(H) == 1)
      k_expert<1><<<grid, NT, smem, st>>>(a);
    else
      k_expert<2><<<grid, NT, smem, st>>>(a);
    prof_end(p, st);
    ++*launches;
    p = prof_begin(h, capturing, 2, st);
    k_reduce<<<dim3((H + NT - 1) / NT, a.R), NT, 0, st>>>(a);
    prof_end(p, st);
    ++*launches;
  }
  return cudaGetLastError();
}

int common_checks(moe_handle* h, const uint16_t* x, int32_t rows, void* ws, size_t ws_bytes) {
  if (!h || !aligned16(x) || !ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_EINVAL;
  if (rows < 1 || rows > h->dims.max_rows) return MOE_EINVAL;
  if (ws_bytes < ws_layout(h->dims, rows).total) return MOE_EWORKSPACE;
  return MOE_OK;
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
  moe_handle* h = new moe_handle();
  h->dims = *dims;
  h->device = device;
  if (cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaMalloc(&h->status, sizeof(unsigned)) != cudaSuccess ||
      cudaMemset(h->status, 0, sizeof(unsigned)) != cudaSuccess) {
    cudaGetLastError();
    if (h->status) cudaFree(h->status);
    delete h;
    return MOE_ECUDA;
  }
  const size_t smem = expert_smem_bytes(dims->hidden);
  cudaError_t e;
  int occ = 0;
  if (nbl_of(dims->hidden) == 1) {
    e = cudaFuncSetAttribute(k_expert<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_expert<1>, NT, smem);
  } else {
    e = cudaFuncSetAttribute(k_expert<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_expert<2>, NT, smem);
  }
  if (e != cudaSuccess || occ < 1) {
    cudaGetLastError();
    cudaFree(h->status);
    delete h;
    return MOE_ECUDA;
  }
  h->expert_ctas_per_sm = occ;
  *out = h;
  return MOE_OK;
}

void moe_destroy(moe_handle* h) {
  if (!h) return;
  DeviceGuard g(h->device);
  if (h->gexec) cudaGraphExecDestroy(h->gexec);
  if (h->status) cudaFree(h->status);
  for (ProfPair& p : h->prof) {
    cudaEventDestroy(p.start);
    cudaEventDestroy(p.stop);
  }
  delete h;
}

int moe_profile(moe_handle* h, int enable) {
  if (!h) return MOE_EINVAL;
  h->profiling = enable != 0;
  h->prof_used = 0;
  return MOE_OK;
}

int moe_profile_read(moe_handle* h, int kind, double* total_ms, int32_t* launches) {
  if (!h || !total_ms || !launches || kind < 0 || kind > 2) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  double t = 0.0;
  int32_t n = 0;
  for (size_t i = 0; i < h->prof_used; ++i) {
    ProfPair& p = h->prof[i];
    if (p.kind != kind) continue;
    if (cudaEventSynchronize(p.stop) != cudaSuccess) return MOE_ECUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, p.start, p.stop) != cudaSuccess) return MOE_ECUDA;
    t += ms;
    ++n;
  }
  *total_ms = t;
  *launches = n;
  return MOE_OK;
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LayerArgs a = make_args(h, w, x_bf16, rows, nullptr, ws);
  a.user_ids = topk_ids;
  a.user_w = topk_w;
  a.user_union = union_ids;
  a.user_nunion = n_union;
  h->last_launches = 0;
  if (cudaMemsetAsync(a.ctrl, 0, sizeof(Ctrl), st) != cudaSuccess) return MOE_ECUDA;
  if (enqueue_layer(h, a, false, st, &h->last_launches) != cudaSuccess) return MOE_ECUDA;
  return MOE_OK;
}

int moe_decode_layer(moe_handle* h, const moe_layer_w* w, const uint16_t* x_bf16, int32_t rows,
                     float* out, void* ws, size_t ws_bytes, void* stream) {
  int rc = common_checks(h, x_bf16, rows, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  if ((rc = check_layer(w)) != MOE_OK) return rc;
  if (!aligned16(out)) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LayerArgs a = make_args(h, w, x_bf16, rows, out, ws);
  h->last_launches = 0;
  if (cudaMemsetAsync(a.ctrl, 0, sizeof(Ctrl), st) != cudaSuccess) return MOE_ECUDA;
  if (enqueue_layer(h, a, true, st, &h->last_launches) != cudaSuccess) return MOE_ECUDA;
  return MOE_OK;
}

static cudaError_t enqueue_round(moe_handle* h, const moe_layer_w* layers, int32_t L,
                                 const uint16_t* x, int32_t rows, float* out, int32_t* stats,
                                 void* ws, cudaStream_t st, int32_t* launches,
                                 bool capturing = false) {
  const size_t HR = (size_t)h->dims.hidden * rows;
  LayerArgs a0 = make_args(h, &layers[0], x, rows, out, ws);
  cudaError_t e = cudaMemsetAsync(a0.ctrl, 0, sizeof(Ctrl), st);
  if (e != cudaSuccess) return e;
  for (int32_t l = 0; l < L; ++l) {
    LayerArgs a = make_args(h, &layers[l], x + (size_t)l * HR, rows, out + (size_t)l * HR, ws);
    a.stats_slot = stats ? stats + l : nullptr;
    e = enqueue_layer(h, a, true, st, launches, capturing);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int moe_round(moe_handle* h, const moe_layer_w* layers, int32_t L, const uint16_t* x_bf16,
              int32_t rows, float* out, int32_t* stats, void* ws, size_t ws_bytes, int use_graph,
              void* stream) {
  int rc = common_checks(h, x_bf16, rows, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  if (!layers || L < 1 || !aligned16(out)) return MOE_EINVAL;
  for (int32_t l = 0; l < L; ++l)
    if ((rc = check_layer(&layers[l])) != MOE_OK) return rc;
  if (use_graph && !stream) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!use_graph) {
    h->last_launches = 0;
    if (enqueue_round(h, layers, L, x_bf16, rows, out, stats, ws, st, &h->last_launches) !=
        cudaSuccess)
      return MOE_ECUDA;
    return MOE_OK;
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
    int32_t n = 0;
    cudaError_t e = enqueue_round(h, layers, L, x_bf16, rows, out, stats, ws, st, &n, true);
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
    h->graph_launches = n;
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

}  // extern "C"
