// GB300 (sm_103a) kernel and C ABI of the MoE layer of a speculative-decoding verify
// round.  See include/moe_verify.h for the operation and the contract.
//
// One persistent cooperative kernel (k_round, one CTA per SM) runs a whole round of L
// layers.  Per layer, with grid-wide barriers B1..B3 in between:
//   P1  router GEMV: this CTA's router rows (staged into shared memory while the
//       previous layer ran: they depend on no data), canonical fp32 order -> logits.
//   B1
//   P2  every CTA reads the logits and builds the same routing in shared memory:
//       per-row top-k (warp per row, redux.sync selection, lower id wins ties),
//       renormalised weights, the ascending expert union U and, per union expert,
//       the (row, rank) pairs that picked it (CSR).
//   P3  gate/up: the U * I units (gate row i + up row i of a union expert) are split
//       contiguously across CTAs by work and streamed through shared-memory slots
//       with 1-D bulk TMA copies; a warp takes one unit of a chunk, for two rows of
//       the expert at a time, and stores h' = w silu(g) v (w the row's routing weight)
//       to the workspace, already in the operand layout the down pass consumes.
//       Meanwhile the down rows of every union expert for this CTA's share of the
//       output rows are prefetched, issued by a warp left without a unit in the first
//       chunk.
//   B2  (every h' written)
//   P4  down: the h' rows come back by bulk copy in waves of up to 8 CSR positions,
//       one warp per position over all of this CTA's output rows o: y = Wd[o] . h'.
//       Each row's y are added in CSR order (its experts ascending) in shared memory
//       -- a fixed order, so a row's output depends only on that row (bitwise),
//       whatever shares the round.
//   B3  (layer l+1's router waits for layer l's output, as a real decode would)
//
// Dequantisation without a convert instruction: a nibble n placed in bits [p, p+4) of
// an otherwise-zero fp32 word is the subnormal n * 2^(p-149); an fma with
// x * 2^(87-4m) (m = the nibble's slot) yields n * x * 2^-62 exactly.  One AND per
// weight (plus one shift per 8), and packed f32x2 FMAs over pairs of weights.  The
// code offset (q = n - 8) is applied once per 32-element block:
// sum (n-8) x = 2^62 acc - 8 sum x.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int NT = 512;  // threads per CTA
constexpr int NW = NT / 32;
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusBadSlot = 2u;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
// device waits count SM cycles: 2 cycles per requested ns bounds the wall time between
// ns (at ~2 GHz) and a few times ns at lower clocks
constexpr long long kCyclesPerNs = 2;
constexpr long long kDefaultWaitCycles = (long long)kDefaultWaitNs * kCyclesPerNs;
constexpr int kPhases = 13;  // phase stamps per layer when profiling (12 intervals)

struct LayerPtrs {
  const float* router;
  const uint8_t* gu_nib;
  const uint16_t* gu_sc;
  const uint8_t* dn_nib;
  const uint16_t* dn_sc;
  const int32_t* slot;  // expert -> bank slot, or null (slot = expert)
  int n_slots;
};

struct RoundArgs {
  int H, E, k, I, R, L;
  int Rmax;  // the handle's max_rows: the shared-memory plan is sized by it, not by R
  int route_only;
  int tail_rank;  // > 0: drop union experts every picking row has at 1-based rank >= it
  const uint16_t* x;  // [L][R][H] bf16 bits
  float* out;         // [L][R][H]
  int* stats;         // [L] |U| per layer, or null
  unsigned* bar;      // [0] barrier arrivals, [33] abort flag
  float* logits;      // [R][E]
  float* hbuf;        // [R*k][I] weighted SwiGLU outputs h' by CSR position, pair layout
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

// Arrival half: the CTA's earlier writes are published by the CTA barrier and the
// release add.  Work that touches nothing other CTAs write may sit between the halves.
__device__ __forceinline__ void grid_arrive(const RoundArgs& a, Sync& sy) {
  __syncthreads();
  sy.epoch += 1;
  if (threadIdx.x == 0) red_release_add(a.bar, 1u);
}

__device__ bool grid_wait(const RoundArgs& a, const Sync& sy) {
  __shared__ int s_ok;
  if (threadIdx.x == 0) {
    const unsigned target = sy.epoch * gridDim.x;
    unsigned* abort_flag = a.bar + 33;
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

__device__ __forceinline__ bool grid_sync(const RoundArgs& a, Sync& sy) {
  grid_arrive(a, sy);
  return grid_wait(a, sy);
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
// The warps share out the (staged router row, activation row) pairs.
__device__ void router_phase(const RoundArgs& a, const uint16_t* x, const float* s_rw) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int NC = a.H >> 7;  // <= 16
  const int n = router_rows_of_cta(a.E);
  // (router row, activation row) pairs over the warps
  for (int pq = warp; pq < n * a.R; pq += NW) {
    const int q = pq / a.R, r = pq - q * a.R;
    const int e = blockIdx.x + gridDim.x * q;
    const float4* wr = reinterpret_cast<const float4*>(s_rw + (size_t)q * a.H) + lane;
    {
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
  int* pos_ui;   // [R*k] union index of the expert at each CSR position
  int* pos_row;  // [R*k] row at each CSR position
  int* slot;     // [E] bank slot of each expert this layer
  int* pick_pos; // [R*k] CSR position of pick (r, j), or -1 if tail-skipped
};

// scratch (inside the staging area, free while routing): mask [E] (zeroed by the
// caller beforehand), off_e [E], ids [R*k], union index [E], best rank [E] (set to
// INT_MAX by the caller beforehand).
//
// Tail skip (Avalon README, "Numbers": experts that every token of a verification
// routes only at rank 7 or lower are skipped): with a.tail_rank = T > 0 an expert whose
// best 1-based rank over the rows that picked it is >= T leaves the union; its picks
// are not evaluated and the other weights are not renormalised.
// It also cuts this CTA's share of the gate/up units into s_range[0..1] (first, end):
// units are shared out by work, a unit of an expert with R_e rows weighing 2 + 2 R_e on
// the fp32 path (a fixed share for the weight stream plus the per-row FMA work; the
// measured chunk times at 1, 2 and 4 rows go about 1 : 1.4 : 2.7) and ceil(R_e / 16) on
// the tensor cores (wide != 0); one row is an even split by count.
// One row without tail skip (E a power of two, 32 <= E <= NT): the whole routing by
// expert-parallel counting, no sequential rounds.  The rank of expert i is the number of
// experts that rank before it (larger logit, or equal logit and lower id), counted over
// quarters of the row by four threads; the k experts of rank < k are the picks (the
// same set and order as select_row), and a ballot over the experts in id order gives
// each pick its union index (the union is the k picks, ascending).  T.w[j] receives
// pick j's logit; softmax_one turns it into the weight.  This CTA's unit range is the
// even split of the k I units.
__device__ __forceinline__ bool route_one_ok(const RoundArgs& a) {
  return a.R == 1 && a.tail_rank == 0 && a.E <= NT && a.E >= 32 && (a.E & (a.E - 1)) == 0;
}

__device__ __forceinline__ int ranks_before_u(unsigned kj, int j, unsigned ki, int i) {
  return (kj > ki || (kj == ki && j < i)) ? 1 : 0;
}

__device__ void route_one(const RoundArgs& a, const Tables& T, unsigned* s_key, int* s_cnt, int* s_wc, int layer,
                          int* s_range) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, E = a.E, k = a.k;
  const int lgE = __ffs(E) - 1, QE = E >> 2;
  if (tid == 0) {
    const unsigned N = (unsigned)k * (unsigned)a.I, G = gridDim.x, c = blockIdx.x;
    s_range[0] = (int)((c * N) / G);
    s_range[1] = (int)(((c + 1) * N) / G);
  }
  unsigned ki = 0;
  if (tid < E) {
    ki = order_key(__ldcg(a.logits + tid));
    s_key[tid] = ki;
  }
  __syncthreads();
  for (int task = tid; task < 4 * E; task += NT) {
    const int q = task >> lgE, i = task & (E - 1), j0 = q * QE;
    const unsigned kv = s_key[i];
    const uint4* row = reinterpret_cast<const uint4*>(s_key + j0);
    int cnt = 0;
    if (j0 + QE <= i || j0 > i) {
      // a quarter wholly below i ranks key j before i when kj >= ki, wholly above when
      // kj > ki (keys of finite logits are >= 1, so kj >= ki is kj > ki - 1)
      const unsigned th = (j0 > i) ? kv : kv - 1u;
#pragma unroll 8
      for (int j4 = 0; j4 < (QE >> 2); ++j4) {
        const uint4 v = row[j4];
        cnt += (v.x > th) + (v.y > th) + (v.z > th) + (v.w > th);
      }
    } else {
#pragma unroll 8
      for (int j4 = 0; j4 < (QE >> 2); ++j4) {
        const uint4 v = row[j4];
        const int j = j0 + 4 * j4;
        cnt += ranks_before_u(v.x, j, kv, i) + ranks_before_u(v.y, j + 1, kv, i) +
               ranks_before_u(v.z, j + 2, kv, i) + ranks_before_u(v.w, j + 3, kv, i);
      }
    }
    s_cnt[task] = cnt;
  }
  __syncthreads();
  const int rank = (tid < E) ? s_cnt[tid] + s_cnt[E + tid] + s_cnt[2 * E + tid] + s_cnt[3 * E + tid] : k;
  const bool picked = rank < k;
  const unsigned b = __ballot_sync(0xffffffffu, picked);
  if (lane == 0) s_wc[warp] = __popc(b);
  __syncthreads();
  int ui = __popc(b & ((1u << lane) - 1u));
  for (int w = 0; w < warp; ++w) ui += s_wc[w];
  if (picked && ui < k) {  // (exactly k are picked unless a logit is NaN, which is undefined)
    T.uni[ui] = tid;
    T.csr_off[ui] = ui;
    T.pos_ui[ui] = ui;
    T.pos_row[ui] = 0;
    T.pair[ui] = rank;
    T.pick_pos[rank] = ui;
    T.w[rank] = key_value(ki);
    if (blockIdx.x == 0) {
      if (a.user_ids) a.user_ids[rank] = tid;
      if (a.user_union) a.user_union[ui] = tid;
    }
  }
  if (tid == 0) {
    T.csr_off[k] = k;
    *T.n_union = k;
    if (blockIdx.x == 0) {
      if (a.user_nunion) *a.user_nunion = k;
      if (a.stats) a.stats[layer] = k;
    }
  }
  __syncthreads();
}

// Weights of route_one's picks (one warp): T.w[j] holds pick j's logit; w_j =
// exp(l_j - l_1) / sum over the k picks, the same warp sum as the general path.
__device__ void softmax_one(const RoundArgs& a, const Tables& T) {
  const int lane = threadIdx.x & 31, k = a.k;
  const float l = (lane < k) ? T.w[lane] : 0.f;
  const float l1 = __shfl_sync(0xffffffffu, l, 0);
  const float ex = (lane < k) ? expf(l - l1) : 0.f;
  const float den = warp_sum(ex);
  if (lane < k) {
    const float w = __fdiv_rn(ex, den);
    T.w[lane] = w;
    if (blockIdx.x == 0 && a.user_w) a.user_w[lane] = w;
  }
}

// Union, CSR tables and this CTA's unit range for rounds of at most 32 picks (no tail
// skip), by one warp: the picks, keyed (expert, row), are sorted across the lanes
// (bitonic network over xor partners); a pick that starts a run of one expert opens a
// union entry, and the ballot of those gives every pick its union index.  Same tables
// and the same unit cut as the general scan below.  s_ids holds the picks' experts.
__device__ void route_small(const RoundArgs& a, const Tables& T, const int* s_ids, int layer, int wide,
                            int* s_range) {
  const int lane = threadIdx.x & 31, k = a.k, P = a.R * k;
  constexpr unsigned FULL = 0xffffffffu;
  const bool live = lane < P;
  unsigned key = live ? ((unsigned)s_ids[lane] << 5) | (unsigned)(lane / k) : FULL;
  int pick = lane;
  // the network over the first NS lanes (NS = the power of two >= P) sorts them
  const int NS = P <= 8 ? 8 : (P <= 16 ? 16 : 32);
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
    if (size > NS) break;
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned ok = __shfl_xor_sync(FULL, key, stride);
      const int op = __shfl_xor_sync(FULL, pick, stride);
      const bool keep_min = ((lane & size) == 0) == ((lane & stride) == 0);
      const bool sw = keep_min ? (ok < key) : (ok > key);
      key = sw ? ok : key;
      pick = sw ? op : pick;
    }
  }
  const int e = (int)(key >> 5), r = (int)(key & 31u);
  const unsigned prev = __shfl_up_sync(FULL, key, 1);
  const bool first = live && (lane == 0 || (prev >> 5) != (key >> 5));
  const unsigned fb = __ballot_sync(FULL, first);
  const int U = __popc(fb);
  const unsigned le = (lane == 31) ? FULL : ((2u << lane) - 1u);
  const int ui = __popc(fb & le) - 1;
  if (live) {
    T.pos_ui[lane] = ui;
    T.pos_row[lane] = r;
    T.pair[lane] = pick;
    T.pick_pos[pick] = lane;
  }
  if (first) {
    T.uni[ui] = e;
    T.csr_off[ui] = lane;
    if (blockIdx.x == 0 && a.user_union) a.user_union[ui] = e;
  }
  if (lane == 0) {
    T.csr_off[U] = P;
    *T.n_union = U;
    if (blockIdx.x == 0) {
      if (a.user_nunion) *a.user_nunion = U;
      if (a.stats) a.stats[layer] = U;
    }
  }
  const int G = gridDim.x, c = blockIdx.x;
  if (a.R == 1) {
    const unsigned N = (unsigned)U * (unsigned)a.I;
    if (lane == 0) {
      s_range[0] = (int)((c * N) / (unsigned)G);
      s_range[1] = (int)(((c + 1) * N) / (unsigned)G);
    }
    return;
  }
  __syncwarp();
  // union expert u = lane: its rows R_e and work weight, prefix over the union
  int wu = 0;
  if (lane < U) {
    const int re = T.csr_off[lane + 1] - T.csr_off[lane];
    wu = wide ? (re + 15) >> 4 : 2 + 2 * re;
  }
  const int lw = a.I * wu;
  int incw = lw;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int tw = __shfl_up_sync(FULL, incw, o);
    if (lane >= o) incw += tw;
  }
  const int wt_total = __shfl_sync(FULL, incw, 31), basew = incw - lw;
  const float wg = (float)wt_total / (float)G;
  const int tgt[2] = {c == 0 ? 0 : min((int)(wg * (float)c), wt_total),
                      c + 1 == G ? wt_total : min((int)(wg * (float)(c + 1)), wt_total)};
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const bool here = lane < U && tgt[q] >= basew && tgt[q] < incw;
    const unsigned owner = __ballot_sync(FULL, here);
    int res = U * a.I;
    if (owner) res = __shfl_sync(FULL, lane * a.I + (tgt[q] - basew) / max(wu, 1), __ffs(owner) - 1);
    if (lane == 0) s_range[q] = res;
  }
}

__device__ int route_phase(const RoundArgs& a, const Tables& T, unsigned* s_mask, int* s_off_e,
                           int* s_ids, int* s_ui, int* s_rank, int layer, int wide, int* s_range) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, k = a.k, R = a.R;
  const bool small = R * k <= 32 && a.tail_rank == 0;
  // route_one's scratch: keys [E] (16-byte aligned: read as uint4), counts [4 E], warp sums
  unsigned* s_key = reinterpret_cast<unsigned*>((reinterpret_cast<uintptr_t>(s_rank + E) + 15) & ~(uintptr_t)15);
  if (route_one_ok(a)) {  // (weights: softmax_one, by the caller)
    route_one(a, T, s_key, reinterpret_cast<int*>(s_key + NT), reinterpret_cast<int*>(s_key + 5 * NT), layer,
              s_range);
    return k;
  }
  // rows: top-k, renormalised weights, row bits of each picked expert
  for (int r = warp; r < R; r += NW) {
    float my_l = 0.f;
    int my_id = 0;
    if (E <= 128)
      select_row<4>(a.logits + (size_t)r * E, E, k, lane, my_l, my_id);
    else  // E <= 512 (moe_create rejects more)
      select_row<16>(a.logits + (size_t)r * E, E, k, lane, my_l, my_id);
    // weights: exp(l_j - l_1) / sum over the k picks (a warp sum: a fixed order per row)
    const float l1 = __shfl_sync(0xffffffffu, my_l, 0);
    const float ex = (lane < k) ? expf(my_l - l1) : 0.f;
    const float den = warp_sum(ex);
    if (lane < k) {
      const float wj = __fdiv_rn(ex, den);
      const int p = r * k + lane;
      s_ids[p] = my_id;
      T.w[p] = wj;
      if (!small) atomicOr(&s_mask[my_id], 1u << r);
      if (a.tail_rank > 0) atomicMin(&s_rank[my_id], lane);
      if (blockIdx.x == 0) {
        if (a.user_ids) a.user_ids[p] = my_id;
        if (a.user_w) a.user_w[p] = wj;
      }
    }
  }
  __syncthreads();
  if (small) {
    if (warp == 0) route_small(a, T, s_ids, layer, wide, s_range);
    __syncthreads();
    return *T.n_union;
  }
  // one warp: exclusive scans over e of (picked ? 1 : 0) and popc(mask) give the union
  // index and the CSR offset of every picked expert (lane l owns a contiguous range)
  if (warp == 0) {
    const int per = (E + 31) >> 5;  // <= 16
    const int e0 = lane * per, e1 = min(e0 + per, E);
    auto weight = [&](unsigned m) { const int re = __popc(m); return wide ? (re + 15) >> 4 : 2 + 2 * re; };
    int lf = 0, lc = 0, lw = 0;
    for (int e = e0; e < e1; ++e) {
      unsigned m = s_mask[e];
      if (m && a.tail_rank > 0 && s_rank[e] + 1 >= a.tail_rank) {
        m = 0u;  // tail-skipped: out of the union, its picks are dropped
        s_mask[e] = 0u;
      }
      lf += (m != 0u);
      lc += __popc(m);
      if (m) lw += a.I * weight(m);
    }
    int incf = lf, incc = lc, incw = lw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int tf = __shfl_up_sync(0xffffffffu, incf, o);
      const int tc = __shfl_up_sync(0xffffffffu, incc, o);
      const int tw = __shfl_up_sync(0xffffffffu, incw, o);
      if (lane >= o) {
        incf += tf;
        incc += tc;
        incw += tw;
      }
    }
    int basef = incf - lf, basec = incc - lc;
    // this CTA's unit range: the targets t(c) ~ c W / G are computed the same way by
    // neighbouring CTAs (in fp32; monotone in c, t(0) = 0, t(G) = W), so the ranges
    // tile the units.
    {
      const int G = gridDim.x, c = blockIdx.x;
      const int U = __shfl_sync(0xffffffffu, incf, 31);
      if (R == 1) {
        const unsigned N = (unsigned)U * (unsigned)a.I;  // < 2^31 (U <= 512, I <= 4096)
        if (lane == 0) {
          s_range[0] = (int)((c * N) / (unsigned)G);
          s_range[1] = (int)(((c + 1) * N) / (unsigned)G);
        }
      } else {
        const int wt_total = __shfl_sync(0xffffffffu, incw, 31), basew = incw - lw;
        const float wg = (float)wt_total / (float)G;
        const int tgt[2] = {c == 0 ? 0 : min((int)(wg * (float)c), wt_total),
                            c + 1 == G ? wt_total : min((int)(wg * (float)(c + 1)), wt_total)};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const bool here = tgt[q] >= basew && tgt[q] < incw;
          int res = U * a.I;
          if (here) {
            int cum = basew, ui = basef;
            for (int e = e0; e < e1; ++e) {
              const unsigned m = s_mask[e];
              if (!m) continue;
              const int w = weight(m), ew = a.I * w;
              if (tgt[q] < cum + ew) {
                res = ui * a.I + (tgt[q] - cum) / w;
                break;
              }
              cum += ew;
              ++ui;
            }
          }
          const unsigned owner = __ballot_sync(0xffffffffu, here);
          res = owner ? __shfl_sync(0xffffffffu, res, __ffs(owner) - 1) : U * a.I;
          if (lane == 0) s_range[q] = res;
        }
      }
    }
    for (int e = e0; e < e1; ++e) {
      const unsigned m = s_mask[e];
      if (m) {
        s_off_e[e] = basec;
        s_ui[e] = basef;
        T.uni[basef] = e;
        T.csr_off[basef] = basec;
        if (blockIdx.x == 0 && a.user_union) a.user_union[basef] = e;
        ++basef;
        basec += __popc(m);
      }
    }
    if (lane == 31) {
      // the last lane's running totals are the union size and the pair count
      *T.n_union = basef;
      T.csr_off[basef] = basec;
      if (blockIdx.x == 0) {
        if (a.user_nunion) *a.user_nunion = basef;
        if (a.stats) a.stats[layer] = basef;
      }
    }
  }
  __syncthreads();
  for (int p = tid; p < R * k; p += NT) {
    const int e = s_ids[p], r = p / k;
    T.pick_pos[p] = -1;
    if (s_mask[e] == 0u) continue;  // (tail-skipped)
    const int pos = s_off_e[e] + __popc(s_mask[e] & ((1u << r) - 1u));
    T.pick_pos[p] = pos;
    T.pair[pos] = p;
    T.pos_row[pos] = r;
    T.pos_ui[pos] = s_ui[e];
  }
  __syncthreads();
  return *T.n_union;
}

// ---------------------------------------------------------------------------------
// P3: gate/up over an even share of the (union expert, intermediate row) units
//
// Unit (ui, i) = gate row i and up row i of union expert ui: H bytes of codes and H/8
// bytes of scales, contiguous in the packed layout.  CTA c owns units
// [c N / G, (c+1) N / G) of the N = U * I units, walked in chunks that stop at expert
// boundaries and at the slot capacity; chunks stream through kGuSlots shared-memory
// slots (1-D bulk copies, one mbarrier per slot).  For every row of the expert a warp
// computes g and v of one unit, lane 0 stores h = silu(g) v to the workspace at
// (CSR position, i).  Down rows of every union expert for this CTA's output rows are
// prefetched into kDnSlots slots meanwhile (they depend only on the routing).

constexpr int kGuSlots = 3;
// gate/up chunks issued before the first one lands (the rest of the ring follows it):
// copies in flight share the bandwidth, so a chunk issued alone arrives sooner
constexpr int kGuFirst = 1;
constexpr int kDnSlots = 11;
// the layer's rows as operand pairs plus block sums (4 rows at hidden 2048), staged once
// per layer when they fit
constexpr size_t kXBytes = 33792;
// Inside the gate/up ring, idle outside the gate/up stream: the next layer's router rows
// at offset 0 (consumed before the routing scratch, also at offset 0, is written) and,
// from kHOffset on, two slots of exchanged h rows for the down pass.
constexpr size_t kHOffset = 32768;
constexpr int kAccStride = 64;  // output rows per CTA are at most this many

struct GuChunk {
  int ui, i0, n;
};

// smem plan: GU ring | DN slots | x pairs | tables | out accumulators | wave outputs |
// chunk list | barriers
struct SmemPlan {
  size_t gu_slot, gu, dn_slot, dn, xrows, uni, csr, pair, w, pos_ui, pos_row, slot, pick, nunion, acc, ybuf,
      chunks, bars, total;
  size_t ring;    // bytes of the gate/up ring (>= kGuSlots * gu_slot)
  size_t h_slot;  // bytes per h slot (two slots from gu + kHOffset)
  int gu_cap;     // units per gate/up chunk
  int h_rows;     // h rows (CSR positions) per h slot
  int max_orows;  // output rows per CTA (ceil(H / grid))
  bool router_fits;
};

__host__ __device__ inline size_t up128(size_t x) { return (x + 127) & ~(size_t)127; }

__host__ __device__ inline SmemPlan smem_plan(int H, int I, int E, int R, int k, int grid) {
  SmemPlan p{};
  const size_t unit = (size_t)H + (size_t)H / 8;
  p.max_orows = (H + grid - 1) / grid;
  p.dn_slot = up128((size_t)p.max_orows * (I / 2)) + up128((size_t)p.max_orows * (I / 16));
  const size_t tables = up128((size_t)E * 4) + up128((size_t)(E + 1) * 4) +
                        5 * up128((size_t)R * k * 4) + up128((size_t)E * 4) + 128 +
                        up128((size_t)R * kAccStride * 4) +
                        up128((size_t)NW * kAccStride * 4) + up128(kGuSlots * 12 + 16) + 256;
  const size_t fixed = tables + kDnSlots * p.dn_slot + kXBytes;
  const size_t limit = (size_t)225 * 1024;
  size_t cap = fixed < limit ? ((limit - fixed) / kGuSlots) / unit : 0;
  if (cap > NW) cap = NW;  // a chunk is one pass of the warps, a unit each
  p.gu_cap = (int)cap;
  p.gu_slot = up128(cap * unit);
  // small shapes: keep room behind kHOffset for full waves of exchanged h rows
  p.ring = kGuSlots * p.gu_slot;
  const size_t want = kHOffset + 2 * up128((size_t)NW * I * 4);
  if (p.ring < want && fixed + want <= limit) p.ring = want;
  size_t off = 0;
  p.gu = off;      off += p.ring;
  p.dn = off;      off += kDnSlots * p.dn_slot;
  p.xrows = off;   off += kXBytes;
  p.uni = off;     off += up128((size_t)E * 4);
  p.csr = off;     off += up128((size_t)(E + 1) * 4);
  p.pair = off;    off += up128((size_t)R * k * 4);
  p.w = off;       off += up128((size_t)R * k * 4);
  p.pos_ui = off;  off += up128((size_t)R * k * 4);
  p.pos_row = off; off += up128((size_t)R * k * 4);
  p.slot = off;    off += up128((size_t)E * 4);
  p.pick = off;    off += up128((size_t)R * k * 4);
  p.nunion = off;  off += 128;
  p.acc = off;     off += up128((size_t)R * kAccStride * 4);
  p.ybuf = off;    off += up128((size_t)NW * kAccStride * 4);
  p.chunks = off;  off += up128(kGuSlots * 12 + 16);
  p.bars = off;    off += 256;
  p.total = off;
  const int rows_per_cta = (E + grid - 1) / grid;
  p.h_slot = p.ring > kHOffset ? ((p.ring - kHOffset) / 2) & ~(size_t)127 : 0;
  p.h_rows = (int)(p.h_slot / ((size_t)I * 4));
  p.router_fits = cap >= 1 && p.max_orows <= kAccStride && p.h_rows >= 1 &&
                  (size_t)rows_per_cta * H * 4 <= kHOffset;
  return p;
}

__device__ void issue_gu_chunk(const RoundArgs& a, const LayerPtrs& W, const Tables& T, uint8_t* dst,
                               uint32_t bar, const GuChunk& c) {
  const size_t H = (size_t)a.H, I = (size_t)a.I;
  const size_t u = (size_t)T.slot[T.uni[c.ui]];
  const size_t first = u * I + (size_t)c.i0;  // unit index within the bank
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(bar, (uint32_t)((size_t)c.n * (H + H / 8)));
  bulk_g2s(smem_u32(dst), W.gu_nib + first * H, (uint32_t)(c.n * H), bar);
  bulk_g2s(smem_u32(dst + (size_t)c.n * H),
           reinterpret_cast<const uint8_t*>(W.gu_sc) + first * (H / 8), (uint32_t)(c.n * (H / 8)), bar);
}

__device__ void issue_dn_chunk(const RoundArgs& a, const LayerPtrs& W, const Tables& T, uint8_t* dst,
                               uint32_t bar, int ui, int o0, int no, size_t codes_room) {
  const size_t H = (size_t)a.H, I = (size_t)a.I;
  const size_t u = (size_t)T.slot[T.uni[ui]];
  const size_t row0 = u * H + (size_t)o0;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(bar, (uint32_t)((size_t)no * (I / 2 + I / 16)));
  bulk_g2s(smem_u32(dst), W.dn_nib + row0 * (I / 2), (uint32_t)(no * (I / 2)), bar);
  bulk_g2s(smem_u32(dst + codes_room), reinterpret_cast<const uint8_t*>(W.dn_sc) + row0 * (I / 16),
           (uint32_t)(no * (I / 16)), bar);
}

// ---------------------------------------------------------------------------------
// Operand pairs.  The word pairs above consume a block's 32 elements as 16 f32x2
// operands: pair p holds elements (16(p/8) + p%8, 16(p/8) + 8 + p%8), pre-scaled by
// slot_scale(p%8).  Activations (once per layer) and exchanged h rows (by their
// producer) are kept in this form, block-interleaved: float4 c of block b (pairs 2c
// and 2c+1) sits at float4 index c * NBlk + b, so lane b's eight 16-byte loads are
// conflict-free.

// Float index of element j of block b in a pair-layout row of NBlk blocks.
__device__ __forceinline__ int pair_index(int b, int j, int NBlk) {
  const int p = ((j >> 4) << 3) | (j & 7);
  return (((p >> 1) * NBlk + b) << 2) | ((p & 1) << 1) | ((j >> 3) & 1);
}

__device__ __forceinline__ void f2unpack(f2_t v, float& lo, float& hi) {
  asm("mov.b64 {%0,%1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// 2^-(exponent of slot_scale(m)): exact inverse of the slot factor.
__device__ __forceinline__ float inv_slot_scale(int m) {
  const int e = (m <= 4) ? 87 - 4 * m : 99 - 4 * m;
  return __int_as_float((127 - e) << 23);
}

// One block of bf16 activations (four 16-byte words, elements 0..31) -> its 16
// operand pairs and -8 times the block sum (summed pair by pair).
__device__ __forceinline__ void convert_block(const uint4 (&u)[4], f2_t (&xp)[16], float& xsum8) {
  float sum = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 ua = u[2 * h], ub = u[2 * h + 1];
    const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float va = (m & 1) ? bf16_hi(wa[m >> 1]) : bf16_lo(wa[m >> 1]);
      const float vb = (m & 1) ? bf16_hi(wb[m >> 1]) : bf16_lo(wb[m >> 1]);
      xp[8 * h + m] = f2pack(va * slot_scale(m), vb * slot_scale(m));
      sum = __fadd_rn(sum, va);
      sum = __fadd_rn(sum, vb);
    }
  }
  xsum8 = -8.f * sum;
}

// This layer's rows as operand pairs in shared memory: s_xp [R][8][NB] float4 and
// s_xs [R][NB] (-8 x block sums).  Done while the router barrier completes.
__device__ void stage_xpairs(const RoundArgs& a, const uint16_t* x, float4* s_xp, float* s_xs) {
  const int NB = a.H >> 5;
  for (int idx = threadIdx.x; idx < a.R * NB; idx += NT) {
    const int r = idx / NB, b = idx - r * NB;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)r * a.H + 32 * b);
    uint4 u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = __ldg(src + i);
    f2_t xp[16];
    float xs;
    convert_block(u, xp, xs);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float a0, a1, b0, b1;
      f2unpack(xp[2 * c], a0, a1);
      f2unpack(xp[2 * c + 1], b0, b1);
      s_xp[((size_t)r * 8 + c) * NB + b] = make_float4(a0, a1, b0, b1);
    }
    s_xs[r * NB + b] = xs;
  }
}

// Operand pairs of block blk of one row: from the staged pairs (XS) or converted from
// the bf16 row in global memory (rows too many to stage).
template <bool XS>
__device__ __forceinline__ void load_xblock(const RoundArgs& a, const uint16_t* x, const float4* s_xp,
                                            const float* s_xs, int row, int blk, f2_t (&xp)[16],
                                            float& xsum8) {
  const int NB = a.H >> 5;
  if (XS) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      // a float4 of pairs is two f32x2 operands as stored: load them as such
      const ulonglong2 f = *reinterpret_cast<const ulonglong2*>(s_xp + ((size_t)row * 8 + c) * NB + blk);
      xp[2 * c] = f.x;
      xp[2 * c + 1] = f.y;
    }
    xsum8 = s_xs[row * NB + blk];
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)row * a.H + 32 * blk);
    uint4 u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = __ldg(src + i);
    convert_block(u, xp, xsum8);
  }
}

// One 32-element block dot for G activation sets: dot[g] = 2^-62 sum n_k x_k.
template <int G>
__device__ __forceinline__ void block_dot(const uint4 nb, const f2_t* const* xp, float* dot) {
  const BlockPairs bp = block_pairs(nb);
  f2_t a0[G], a1[G];
#pragma unroll
  for (int g = 0; g < G; ++g) a0[g] = a1[g] = 0ull;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const f2_t e0 = slot_pair(bp, 0, m), e1 = slot_pair(bp, 1, m);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      ffma2(a0[g], e0, xp[g][m]);
      ffma2(a1[g], e1, xp[g][8 + m]);
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) dot[g] = __fadd_rn(f2sum(a0[g]), f2sum(a1[g]));
}

// V values per lane (V a power of two <= 16) summed over the warp; value v ends in
// lanes [v 32/V, (v+1) 32/V).  Each value is summed over the same xor tree of lane bits
// 4..0 as warp_sum (only the operand order of commutative adds differs), so its result
// does not depend on the slot it travels in.
template <int V>
__device__ __forceinline__ float warp_sum_multi(float (&v)[V], int lane) {
  constexpr int LOGV = (V >= 16) ? 4 : (V >= 8) ? 3 : (V >= 4) ? 2 : (V >= 2) ? 1 : 0;
  static_assert((1 << LOGV) == V, "V must be a power of two <= 16");
#pragma unroll
  for (int s = 0; s < LOGV; ++s) {
    const int n = V >> s, o = 16 >> s;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
    }
  }
  float s = v[0];
#pragma unroll
  for (int o = 16 >> LOGV; o >= 1; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
  return s;
}

// Gate/up of unit t of chunk c for the rows at CSR positions pp .. pp+G-1: per lane
// its NBL blocks of the gate and up rows, one multi-value reduction, then the lane
// holding a row's gate value takes the up value from the next lane group and stores
// h' = w silu(g) v, pre-scaled, in pair layout.
template <int NBL, int G, bool XS>
__device__ __forceinline__ void gateup_unit(const RoundArgs& a, const Tables& T, const uint8_t* slot,
                                            const GuChunk& c, int t, int pp, const uint16_t* x,
                                            const float4* s_xp, const float* s_xs) {
  const int H = a.H, NB = H >> 5;
  const int lane = threadIdx.x & 31;
  int row[G];
#pragma unroll
  for (int g = 0; g < G; ++g) row[g] = T.pos_row[pp + g];
  const uint8_t* codes = slot;
  const uint16_t* scales = reinterpret_cast<const uint16_t*>(slot + (size_t)c.n * H);
  constexpr int V = 2 * G;  // value 2 g + wrow
  float v[V];
#pragma unroll
  for (int i = 0; i < V; ++i) v[i] = 0.f;
  const int sw = (c.i0 + t) & 7;
#pragma unroll
  for (int tb = 0; tb < NBL; ++tb) {
    const int blk = lane + 32 * tb;
    if (blk < NB) {
      f2_t xp[G][16];
      float xsum8[G];
#pragma unroll
      for (int g = 0; g < G; ++g) load_xblock<XS>(a, x, s_xp, s_xs, row[g], blk, xp[g], xsum8[g]);
      const f2_t* xps[G];
#pragma unroll
      for (int g = 0; g < G; ++g) xps[g] = xp[g];
#pragma unroll
      for (int wrow = 0; wrow < 2; ++wrow) {
        // unit t of the chunk is intermediate row i0 + t of the expert: its blocks sit at
        // blk ^ ((i0 + t) & 7), gate and up alike
        const size_t w = (size_t)(t * 2 + wrow) * NB + (blk ^ sw);
        const uint4 nb = *reinterpret_cast<const uint4*>(codes + w * 16);
        const float sc = half_bits(scales[w]);
        float dot[G];
        block_dot<G>(nb, xps, dot);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float& acc = v[2 * g + wrow];
          acc = __fmaf_rn(sc, __fmaf_rn(dot[g], 0x1p62f, xsum8[g]), acc);
        }
      }
    }
  }
  const float s = warp_sum_multi<V>(v, lane);
  constexpr int LPV = 32 / V;  // lanes per value
  const float up = __shfl_down_sync(0xffffffffu, s, LPV);
  const int vi = lane / LPV;
  if ((lane % LPV) == 0 && (vi & 1) == 0) {
    const int g = vi >> 1;
    const int i = c.i0 + t, j = i & 31;
    const int pair = T.pair[pp + g];
    const float hh = __fmul_rn(__fdiv_rn(s, __fadd_rn(1.f, expf(-s))), up);
    const float hw = __fmul_rn(T.w[pair], hh);
    a.hbuf[(size_t)(pp + g) * a.I + pair_index(i >> 5, j, a.I >> 5)] = hw * slot_scale(j & 7);
  }
}

// Gate/up of one staged chunk (at most NW units): warp w takes unit w, the rows of the
// expert two at a time when the activations are staged.
template <int NBL, bool XS>
__device__ __forceinline__ void gateup_chunk(const RoundArgs& a, const Tables& T, const uint8_t* slot,
                                             const GuChunk& c, const uint16_t* x, const float4* s_xp,
                                             const float* s_xs) {
  const int warp = threadIdx.x >> 5;
  const int p0 = T.csr_off[c.ui], p1 = T.csr_off[c.ui + 1];
  for (int t = warp; t < c.n; t += NW) {
    int pp = p0;
    if (XS)  // (converting two rows from global memory at once would not fit the registers)
      for (; pp + 1 < p1; pp += 2) gateup_unit<NBL, 2, XS>(a, T, slot, c, t, pp, x, s_xp, s_xs);
    for (; pp < p1; ++pp) gateup_unit<NBL, 1, XS>(a, T, slot, c, t, pp, x, s_xp, s_xs);
  }
}

// Gate/up of one staged chunk when the round has one row: the operand pairs of each
// lane's first block of the row (xr) stay in registers for the whole layer, so a unit
// reads only its codes, scales and the second block's pairs from shared memory (both
// blocks in registers would not fit beside the rest of the kernel).  Same operations in
// the same order as gateup_unit with one row, so the results are the same bits.
template <int NBL>
__device__ __forceinline__ void gateup_chunk_r1(const RoundArgs& a, const Tables& T, const uint8_t* slot,
                                                const GuChunk& c, const f2_t (&xr)[16], const float4* s_xp,
                                                const float* s_xs) {
  const int H = a.H, NB = H >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pp = T.csr_off[c.ui];
  const uint8_t* codes = slot;
  const uint16_t* scales = reinterpret_cast<const uint16_t*>(slot + (size_t)c.n * H);
  for (int t = warp; t < c.n; t += NW) {
    float v[2] = {0.f, 0.f};
    const int sw = (c.i0 + t) & 7;
#pragma unroll
    for (int tb = 0; tb < NBL; ++tb) {
      const int blk = lane + 32 * tb;
      if (blk < NB) {
        f2_t xq[16];
        float xs;
        if (tb == 0) {
#pragma unroll
          for (int m = 0; m < 16; ++m) xq[m] = xr[m];
          xs = s_xs[blk];
        } else {
          load_xblock<true>(a, nullptr, s_xp, s_xs, 0, blk, xq, xs);
        }
        const f2_t* xps[1] = {xq};
#pragma unroll
        for (int wrow = 0; wrow < 2; ++wrow) {
          const size_t w = (size_t)(t * 2 + wrow) * NB + (blk ^ sw);
          const uint4 nb = *reinterpret_cast<const uint4*>(codes + w * 16);
          const float sc = half_bits(scales[w]);
          float dot[1];
          block_dot<1>(nb, xps, dot);
          v[wrow] = __fmaf_rn(sc, __fmaf_rn(dot[0], 0x1p62f, xs), v[wrow]);
        }
      }
    }
    const float s = warp_sum_multi<2>(v, lane);
    const float up = __shfl_down_sync(0xffffffffu, s, 16);
    if (lane == 0) {
      const int i = c.i0 + t, j = i & 31;
      const int pair = T.pair[pp];
      const float hh = __fmul_rn(__fdiv_rn(s, __fadd_rn(1.f, expf(-s))), up);
      const float hw = __fmul_rn(T.w[pair], hh);
      a.hbuf[(size_t)pp * a.I + pair_index(i >> 5, j, a.I >> 5)] = hw * slot_scale(j & 7);
    }
  }
}

// ---------------------------------------------------------------------------------
// P4: this CTA's output rows [o0, o0 + no), a wave of CSR positions at a time

// y of one CSR position over this CTA's output rows [ob0, ob1): the position's h' row
// (pair layout, shared memory) against each output row's down codes of its expert;
// y[ol] to s_yw.  Lanes >= I/32 hold no block.
__device__ __forceinline__ void down_position(const RoundArgs& a, const uint8_t* dslot, size_t codes_room,
                                              int o0, int ob0, int ob1, const float4* s_h, float* s_yw) {
  const int NBI = a.I >> 5;
  const int lane = threadIdx.x & 31;
  f2_t hp[16];
  float hsum8 = 0.f;
  if (lane < NBI) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const ulonglong2 f = *reinterpret_cast<const ulonglong2*>(s_h + c * NBI + lane);
      hp[2 * c] = f.x;
      hp[2 * c + 1] = f.y;
    }
    // -8 x the block sum of h', undoing each slot's power-of-two factor exactly
    float sum = 0.f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      float a0, a1, b0, b1;
      f2unpack(hp[m], a0, a1);
      f2unpack(hp[8 + m], b0, b1);
      sum = __fmaf_rn(__fadd_rn(__fadd_rn(a0, a1), __fadd_rn(b0, b1)), inv_slot_scale(m), sum);
    }
    hsum8 = -8.f * sum;
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) hp[i] = 0ull;
  }
  const uint8_t* codes = dslot;
  const uint16_t* scales = reinterpret_cast<const uint16_t*>(dslot + codes_room);
  const f2_t* hps[1] = {hp};
  // rows in groups of DG, one multi-value reduction per group
  constexpr int DG = 8;
  for (int ob = ob0; ob < ob1; ob += DG) {
    float part[DG];
#pragma unroll
    for (int jj = 0; jj < DG; ++jj) {
      part[jj] = 0.f;
      const int ol = ob + jj;
      if (lane < NBI && ol < ob1) {
        const int pos = block_pos(lane, o0 + ol);
        const uint4 nb = *reinterpret_cast<const uint4*>(codes + ((size_t)ol * NBI + pos) * 16);
        const float sc = half_bits(scales[ol * NBI + pos]);
        float dot[1];
        block_dot<1>(nb, hps, dot);
        part[jj] = __fmul_rn(sc, __fmaf_rn(dot[0], 0x1p62f, hsum8));
      }
    }
    const float y = warp_sum_multi<DG>(part, lane);
    constexpr int LPV = 32 / DG;
    if ((lane % LPV) == 0 && ob + lane / LPV < ob1) s_yw[ob + lane / LPV] = y;
  }
}

// ---------------------------------------------------------------------------------
// Wide verify rounds (at least kMmaRows rows): gate/up and down on the tensor cores
// (mma.sync m16n8k16, bf16 operands, fp32 accumulation).
//
// A nibble n in the low four bits of a bf16 whose other bits are those of 128.0 is the
// bf16 value 128 + n, exactly; one mask-and-or per pair of weights (two nibbles 16 bits
// apart land in the two halves of a bf16x2 register), and one bf16x2 subtraction of 136
// gives n - 8, again exactly.  Inside each 32-element block the MMA's k order is
// permuted so that thread t's A fragments for the block's two k16 steps are exactly
// the eight nibbles of 32-bit word t of a row's 16-byte block:
//   step 0: k (2t, 2t+1) <- elements (8t, 8t+4),   k (2t+8, 2t+9) <- (8t+1, 8t+5)
//   step 1: k (2t, 2t+1) <- (8t+2, 8t+6),          k (2t+8, 2t+9) <- (8t+3, 8t+7)
// The B fragments (activations, or the exchanged h' split into bf16 hi + lo) follow the
// same permutation.  A block's MMAs give sum (n - 8) b, which the block scale then
// multiplies into the fp32 accumulator.  Each warp keeps one A tile (16 weight rows x
// one K part) in registers for up to two n-tiles (16 expert rows or positions).  Every
// tile's K range is split in the same fixed parts whatever the other rows are, and the
// parts are added in a fixed order, so a row's result does not depend on the rows it
// shares the round with.

constexpr int kMmaRows = 8;
constexpr int kKPartsGu = 8;  // K parts of a gate/up tile (hidden blocks)
constexpr int kKPartsDn = 4;  // K parts of a down tile (intermediate blocks)
static_assert(NW % kKPartsGu == 0 && NW % kKPartsDn == 0, "a tile's K parts run in one round");
// scratch of the tensor-core path inside the activation-pair region (unused then)
constexpr int kMmaMaxPos = 256;          // CSR positions (rows x top-k) of a wide round
constexpr size_t kMmaPart = 0;           // [NW][2][16][8] fp32 partial tiles
constexpr size_t kMmaY = (size_t)NW * 256 * 4;  // [kMmaMaxPos][16] fp32: y per position and output row
static_assert(kMmaY + (size_t)kMmaMaxPos * 16 * 4 <= kXBytes, "wide scratch fits the activation region");


// Gate/up of one staged chunk on the tensor cores.  A tile = 8 units of the chunk (A
// row g: the gate row of unit g, row g + 8: its up row, so the eight lanes' rows have
// eight different block swizzles) x up to 16 of the expert's rows (two n-tiles) x one
// of kKPartsGu K parts; one warp per tile part.  The parts are added in order, then
// h' = w silu(g) v is stored split into bf16 hi + lo in the down pass's fragment order.
__device__ void gateup_chunk_mma(const RoundArgs& a, const Tables& T, const uint8_t* slot, const GuChunk& c,
                                 const uint16_t* x, float* s_part) {
  const int H = a.H, NB = H >> 5, NBI = a.I >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int p0 = T.csr_off[c.ui], Re = T.csr_off[c.ui + 1] - p0;
  const int NTP = (Re + 15) >> 4, MT = (c.n + 7) >> 3, n_asg = MT * NTP * kKPartsGu;
  const uint8_t* codes = slot;
  const uint16_t* scales = reinterpret_cast<const uint16_t*>(slot + (size_t)c.n * H);
  uint16_t* hb = reinterpret_cast<uint16_t*>(a.hbuf);
  for (int j0 = 0; j0 < n_asg; j0 += NW) {
    const int j = j0 + warp;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (j < n_asg) {
      const int gi = j / kKPartsGu, kp = j - gi * kKPartsGu;
      const int mt = gi / NTP, ntp = gi - mt * NTP;
      // units past the chunk repeat its last one; their results are dropped
      const int u = min(mt * 8 + g, c.n - 1), kk = (c.i0 + u) & 7;
      const uint32_t* wg = reinterpret_cast<const uint32_t*>(codes + (size_t)(2 * u) * NB * 16) + t;
      const uint32_t* wu = wg + NB * 4;
      const uint16_t* sg_ = scales + (size_t)(2 * u) * NB;
      const uint16_t* su_ = sg_ + NB;
      // columns past the expert's rows repeat its last row; their results are dropped
      const int c0 = ntp * 16 + g;
      const bool two = ntp * 16 + 8 < Re;
      const uint4* x0 = reinterpret_cast<const uint4*>(x + (size_t)T.pos_row[p0 + min(c0, Re - 1)] * H) + t;
      const uint4* x1 = reinterpret_cast<const uint4*>(x + (size_t)T.pos_row[p0 + min(c0 + 8, Re - 1)] * H) + t;
      const int b0 = (kp * NB) / kKPartsGu, b1 = ((kp + 1) * NB) / kKPartsGu;
#pragma unroll 2
      for (int b = b0; b < b1; ++b) {
        const int pb = b ^ kk;
        uint32_t pg[4], pu[4];
        dq_word(wg[4 * pb], pg);
        dq_word(wu[4 * pb], pu);
        const float sg = half_bits(sg_[pb]), su = half_bits(su_[pb]);
        {
          uint32_t bf[4];
          bfrag_x(__ldg(x0 + 4 * b), bf);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16(d, pg[0], pu[0], pg[1], pu[1], bf[0], bf[1]);
          mma_bf16(d, pg[2], pu[2], pg[3], pu[3], bf[2], bf[3]);
          acc[0][0] = __fmaf_rn(sg, d[0], acc[0][0]);
          acc[0][1] = __fmaf_rn(sg, d[1], acc[0][1]);
          acc[0][2] = __fmaf_rn(su, d[2], acc[0][2]);
          acc[0][3] = __fmaf_rn(su, d[3], acc[0][3]);
        }
        if (two) {
          uint32_t bf[4];
          bfrag_x(__ldg(x1 + 4 * b), bf);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16(d, pg[0], pu[0], pg[1], pu[1], bf[0], bf[1]);
          mma_bf16(d, pg[2], pu[2], pg[3], pu[3], bf[2], bf[3]);
          acc[1][0] = __fmaf_rn(sg, d[0], acc[1][0]);
          acc[1][1] = __fmaf_rn(sg, d[1], acc[1][1]);
          acc[1][2] = __fmaf_rn(su, d[2], acc[1][2]);
          acc[1][3] = __fmaf_rn(su, d[3], acc[1][3]);
        }
      }
    }
    store_part(s_part + warp * 256, acc, g, t);
    __syncthreads();
    for (int i = threadIdx.x; i < (NW / kKPartsGu) * 128; i += NT) {
      const int gl = i >> 7, nt = (i >> 6) & 1, uu = (i >> 3) & 7, cc = i & 7;
      const int gi = j0 / kKPartsGu + gl;
      if (gi >= MT * NTP) continue;
      const int mt = gi / NTP, ntp = gi - mt * NTP;
      const int u = mt * 8 + uu, col = ntp * 16 + nt * 8 + cc;
      if (u >= c.n || col >= Re) continue;
      float gs = 0.f, vs = 0.f;
#pragma unroll
      for (int kp = 0; kp < kKPartsGu; ++kp) {
        const float* P = s_part + (gl * kKPartsGu + kp) * 256 + nt * 128;
        gs = __fadd_rn(gs, P[uu * 8 + cc]);
        vs = __fadd_rn(vs, P[64 + uu * 8 + cc]);
      }
      const int pp = p0 + col;
      const float hh = __fmul_rn(__fdiv_rn(gs, __fadd_rn(1.f, expf(-gs))), vs);
      const float hw = __fmul_rn(T.w[T.pair[pp]], hh);
      const __nv_bfloat16 hi = __float2bfloat16_rn(hw);
      const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(hw, __bfloat162float(hi)));
      const int i2 = c.i0 + u, jj = i2 & 31, e = jj & 7;
      const size_t base = (((size_t)pp * NBI + (i2 >> 5)) * 4 + (jj >> 3)) * 16 + 2 * (e & 3) + (e >> 2);
      hb[base] = __bfloat16_as_ushort(hi);
      hb[base + 8] = __bfloat16_as_ushort(lo);
    }
    __syncthreads();
  }
}

// One round of the wide down pass on the tensor cores: NW tile parts.  Assignment j ->
// position group j / kKPartsDn (group = up to 16 consecutive CSR positions of one
// expert: `gpe` groups per expert) and K part j % kKPartsDn; a tile = this CTA's output
// rows (at most 16) x the group's positions (two n-tiles).  B = h' (hi + lo bf16,
// fragment order) read from the workspace through L2, two MMAs per k16 step and n-tile.
// y[position][output row] -> s_yall.
__device__ void down_round_mma(const RoundArgs& a, const Tables& T, const uint8_t* dn, size_t dn_slot,
                               size_t codes_room, int o0, int no, int j0, int n_asg, int gpe, float* s_part,
                               float* s_yall) {
  const int NBI = a.I >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const uint8_t* hb = reinterpret_cast<const uint8_t*>(a.hbuf);
  const int j = j0 + warp;
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  if (j < n_asg) {
    const int gi = j / kKPartsDn, kp = j - gi * kKPartsDn;
    const int ui = gi / gpe, p0 = T.csr_off[ui] + 16 * (gi - ui * gpe);
    const int cnt = min(16, T.csr_off[ui + 1] - p0);
    if (cnt > 0) {
      const uint8_t* codes = dn + (size_t)(ui % kDnSlots) * dn_slot;
      const uint16_t* scales = reinterpret_cast<const uint16_t*>(codes + codes_room);
      // output rows past this CTA's repeat its last one; their results are dropped
      const int ra = min(g, no - 1), rb = min(g + 8, no - 1);
      const int ka = (o0 + ra) & 7, kb = (o0 + rb) & 7;
      const uint32_t* wa_ = reinterpret_cast<const uint32_t*>(codes + (size_t)ra * NBI * 16) + t;
      const uint32_t* wb_ = reinterpret_cast<const uint32_t*>(codes + (size_t)rb * NBI * 16) + t;
      const uint16_t* sa_ = scales + (size_t)ra * NBI;
      const uint16_t* sb_ = scales + (size_t)rb * NBI;
      // columns past the group's positions repeat its last one; their results are dropped
      const bool two = cnt > 8;
      const uint4* h0 = reinterpret_cast<const uint4*>(hb + (size_t)(p0 + min(g, cnt - 1)) * NBI * 128) + 2 * t;
      const uint4* h1 = reinterpret_cast<const uint4*>(hb + (size_t)(p0 + min(g + 8, cnt - 1)) * NBI * 128) + 2 * t;
      const int b0 = (kp * NBI) / kKPartsDn, b1 = ((kp + 1) * NBI) / kKPartsDn;
#pragma unroll 2
      for (int b = b0; b < b1; ++b) {
        const int pa = b ^ ka, pb = b ^ kb;
        uint32_t fa[4], fb[4];
        dq_word(wa_[4 * pa], fa);
        dq_word(wb_[4 * pb], fb);
        const float sa = half_bits(sa_[pa]), sb = half_bits(sb_[pb]);
        {
          const uint4 hi = __ldcg(h0 + 8 * b), lo = __ldcg(h0 + 8 * b + 1);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16(d, fa[0], fb[0], fa[1], fb[1], hi.x, hi.y);
          mma_bf16(d, fa[0], fb[0], fa[1], fb[1], lo.x, lo.y);
          mma_bf16(d, fa[2], fb[2], fa[3], fb[3], hi.z, hi.w);
          mma_bf16(d, fa[2], fb[2], fa[3], fb[3], lo.z, lo.w);
          acc[0][0] = __fmaf_rn(sa, d[0], acc[0][0]);
          acc[0][1] = __fmaf_rn(sa, d[1], acc[0][1]);
          acc[0][2] = __fmaf_rn(sb, d[2], acc[0][2]);
          acc[0][3] = __fmaf_rn(sb, d[3], acc[0][3]);
        }
        if (two) {
          const uint4 hi = __ldcg(h1 + 8 * b), lo = __ldcg(h1 + 8 * b + 1);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16(d, fa[0], fb[0], fa[1], fb[1], hi.x, hi.y);
          mma_bf16(d, fa[0], fb[0], fa[1], fb[1], lo.x, lo.y);
          mma_bf16(d, fa[2], fb[2], fa[3], fb[3], hi.z, hi.w);
          mma_bf16(d, fa[2], fb[2], fa[3], fb[3], lo.z, lo.w);
          acc[1][0] = __fmaf_rn(sa, d[0], acc[1][0]);
          acc[1][1] = __fmaf_rn(sa, d[1], acc[1][1]);
          acc[1][2] = __fmaf_rn(sb, d[2], acc[1][2]);
          acc[1][3] = __fmaf_rn(sb, d[3], acc[1][3]);
        }
      }
    }
  }
  store_part(s_part + warp * 256, acc, g, t);
  __syncthreads();
  for (int i = threadIdx.x; i < (NW / kKPartsDn) * 256; i += NT) {
    const int gl = i >> 8, nt = (i >> 7) & 1, r = (i >> 3) & 15, cc = i & 7;
    const int gi = j0 / kKPartsDn + gl;
    if (gi * kKPartsDn >= n_asg || r >= no) continue;
    const int ui = gi / gpe, p0 = T.csr_off[ui] + 16 * (gi - ui * gpe);
    const int pos = nt * 8 + cc;
    if (pos >= T.csr_off[ui + 1] - p0) continue;
    float y = 0.f;
#pragma unroll
    for (int kp = 0; kp < kKPartsDn; ++kp) y = __fadd_rn(y, s_part[(gl * kKPartsDn + kp) * 256 + nt * 128 + r * 8 + cc]);
    s_yall[(p0 + pos) * 16 + r] = y;
  }
  __syncthreads();
}

// Exchanged h rows of CSR positions [pa, pb) (contiguous in the workspace) -> slot.
__device__ __forceinline__ void issue_hbatch(const RoundArgs& a, uint8_t* dst, uint32_t bar, int pa, int pb) {
  const size_t bytes = (size_t)(pb - pa) * a.I * 4;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(bar, (uint32_t)bytes);
  bulk_g2s(smem_u32(dst), a.hbuf + (size_t)pa * a.I, (uint32_t)bytes, bar);
}

// Leaving early: gives every copy still in flight a bounded chance to land (so no bulk
// copy targets shared memory of an exited CTA) and raises the abort flag.  Out of line:
// it never runs on the normal path.
__device__ __noinline__ void drain_and_abort(const RoundArgs& a, const uint64_t* bars, unsigned gu_pend,
                                             unsigned gu_ph, unsigned dn_pend, unsigned dn_ph,
                                             unsigned h_pend, unsigned h_ph, bool router_pend,
                                             unsigned ph_router) {
  for (int q = 0; q < kGuSlots; ++q)
    if (gu_pend & (1u << q))
      mbar_wait_bounded(smem_u32(bars + q), (gu_ph >> q) & 1u, a.status, kDefaultWaitCycles);
  for (int q = 0; q < kDnSlots; ++q)
    if (dn_pend & (1u << q))
      mbar_wait_bounded(smem_u32(bars + kGuSlots + q), (dn_ph >> q) & 1u, a.status, kDefaultWaitCycles);
  for (int q = 0; q < 2; ++q)
    if (h_pend & (1u << q))
      mbar_wait_bounded(smem_u32(bars + kGuSlots + kDnSlots + 1 + q), (h_ph >> q) & 1u, a.status,
                        kDefaultWaitCycles);
  if (router_pend)
    mbar_wait_bounded(smem_u32(bars + kGuSlots + kDnSlots), ph_router, a.status, kDefaultWaitCycles);
  if (threadIdx.x == 0) atomicExch(a.bar + 33, 1u);
}

// NBL: 32-element blocks per lane along H (1 up to H 1024, 2 above).  WIDE: the round
// has enough rows for the tensor-core gate/up and down (wide_round() on the host).
template <int NBL, bool WIDE>
__global__ void __launch_bounds__(NT, 1) k_round(const __grid_constant__ RoundArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = gridDim.x;
  const SmemPlan P = smem_plan(a.H, a.I, a.E, a.Rmax, a.k, G);
  // mbarriers: kGuSlots GU slots, kDnSlots DN slots, the router rows, two h slots
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bars);
  const int bar_dn0 = kGuSlots, bar_h0 = kGuSlots + kDnSlots + 1;
  const uint32_t bar_router = smem_u32(bars + kGuSlots + kDnSlots);
  uint8_t* gu = smem + P.gu;
  uint8_t* dn = smem + P.dn;
  float4* s_xp = reinterpret_cast<float4*>(smem + P.xrows);
  float* s_xs = reinterpret_cast<float*>(smem + P.xrows + (size_t)a.R * a.H * 4);
  constexpr bool mma = WIDE;  // tensor-core gate/up and down
  const bool x_staged = !mma && (size_t)a.R * a.H * 4 + (size_t)a.R * (a.H >> 5) * 4 <= kXBytes;
  float* s_mpart = reinterpret_cast<float*>(smem + P.xrows + kMmaPart);
  float* s_yall = reinterpret_cast<float*>(smem + P.xrows + kMmaY);
  float* s_rw = reinterpret_cast<float*>(gu);
  float* s_acc = reinterpret_cast<float*>(smem + P.acc);
  float* s_y = reinterpret_cast<float*>(smem + P.ybuf);
  GuChunk* s_chunks = reinterpret_cast<GuChunk*>(smem + P.chunks);
  Tables T{reinterpret_cast<int*>(smem + P.uni),     reinterpret_cast<int*>(smem + P.csr),
           reinterpret_cast<int*>(smem + P.pair),    reinterpret_cast<float*>(smem + P.w),
           reinterpret_cast<int*>(smem + P.nunion),  reinterpret_cast<int*>(smem + P.pos_ui),
           reinterpret_cast<int*>(smem + P.pos_row), reinterpret_cast<int*>(smem + P.slot),
           reinterpret_cast<int*>(smem + P.pick)};
  // routing scratch lives in the (then idle) gate/up ring
  unsigned* s_mask = reinterpret_cast<unsigned*>(gu);
  int* s_off_e = reinterpret_cast<int*>(gu + (size_t)a.E * 4);
  int* s_ids = reinterpret_cast<int*>(gu + (size_t)a.E * 8);
  int* s_ui = reinterpret_cast<int*>(gu + (size_t)a.E * 8 + (size_t)a.R * a.k * 4);
  int* s_rank = s_ui + a.E;
  if (tid == 0) {
    for (int i = 0; i < bar_h0 + 2; ++i) mbar_init(smem_u32(bars + i), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    issue_router_rows(a, a.layer[0].router, s_rw, bar_router);
  }
  __syncthreads();
  unsigned ph_router = 0u;
  bool router_pend = router_rows_of_cta(a.E) > 0;  // layer 0's rows are in flight
  Sync sy;
  unsigned gu_ph = 0u, gu_pend = 0u;  // bit q: parity / in flight, GU slot q
  unsigned dn_ph = 0u, dn_pend = 0u;  // bit q: parity / in flight, DN slot q
  unsigned h_ph = 0u, h_pend = 0u;    // bit q: parity / in flight, h slot q
  auto bail = [&]() {
    drain_and_abort(a, bars, gu_pend, gu_ph, dn_pend, dn_ph, h_pend, h_ph, router_pend, ph_router);
  };
  // waits for one mbarrier phase with every thread; false (after bail) if it gave up
  auto wait_all = [&](int bi, unsigned& ph, unsigned& pend, int q) -> bool {
    const bool ok = mbar_wait_bounded(smem_u32(bars + bi), (ph >> q) & 1u, a.status, a.wait_cycles);
    if (__syncthreads_or(!ok)) {
      bail();
      return false;
    }
    ph ^= 1u << q;
    pend &= ~(1u << q);
    return true;
  };
  const size_t RH = (size_t)a.R * a.H;
  const int o0 = (int)(((long long)blockIdx.x * a.H) / G);
  const int no = (int)(((long long)(blockIdx.x + 1) * a.H) / G) - o0;
  const size_t codes_room = up128((size_t)P.max_orows * (a.I / 2));
  // CSR positions per down wave: at most one per warp, per h-slot row, and per DN slot
  // (a wave spans at most WV experts, all inside the window of issued DN slots)
  const int WV = min(min(P.h_rows, NW), kDnSlots);
  auto hslot = [&](int q) { return gu + kHOffset + (size_t)q * P.h_slot; };
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
    // B1 (all logits written); the activation pairs are built while it completes
    grid_arrive(a, sy);
    for (int e = tid; e < a.E; e += NT) {  // (the router rows there are consumed)
      s_mask[e] = 0u;
      s_rank[e] = INT_MAX;
      // this layer's expert -> slot table (ingress data); an entry outside the bank is
      // reported and replaced by slot 0, so no copy leaves the bank
      int sl = e;
      if (W.slot) {
        sl = __ldg(W.slot + e);
        if ((unsigned)sl >= (unsigned)W.n_slots) {
          atomicOr(a.status, kStatusBadSlot);
          sl = 0;
        }
      }
      T.slot[e] = sl;
    }
    if (x_staged && !a.route_only) stage_xpairs(a, x, s_xp, s_xs);
    if (!grid_wait(a, sy)) {
      bail();
      return;
    }
    stamp(a, l, 2);
    int* s_range = reinterpret_cast<int*>(smem + P.chunks + kGuSlots * 12 + 20);
    const int U = route_phase(a, T, s_mask, s_off_e, s_ids, s_ui, s_rank, l, mma ? 1 : 0, s_range);
    stamp(a, l, 3);
    const bool one = route_one_ok(a);  // the picks' weights are still to be computed
    if (a.route_only) {
      if (one && warp == 1) softmax_one(a, T);
      return;
    }
    // ---- this CTA's share of the gate/up units (cut during routing); chunks issued
    // through the ring: thread 0 cuts them lazily (stopping at expert boundaries and the
    // slot size) and leaves the descriptor of chunk n in ring entry n % kGuSlots when it
    // issues it ----
    // thread 0's chunk cursor lives in shared memory (cur, end, expert, offset), so no
    // thread carries it in registers through the gate/up loop
    int* s_cursor = reinterpret_cast<int*>(smem + P.chunks + kGuSlots * 12 + 4);
    // on the CUDA-core path the first chunk leaves the last warp without a unit: that
    // warp issues the rest of the ring and the down prefetch while the others compute
    const int cap0 = mma ? P.gu_cap : min(P.gu_cap, NW - 1);
    auto next_chunk = [&](int cap) {
      int cur = s_cursor[0], ui = s_cursor[2], i0 = s_cursor[3];
      int nn = s_cursor[1] - cur;
      if (nn > a.I - i0) nn = a.I - i0;
      if (nn > cap) nn = cap;
      const GuChunk ch{ui, i0, nn};
      cur += nn;
      i0 += nn;
      if (i0 == a.I) {
        ++ui;
        i0 = 0;
      }
      s_cursor[0] = cur;
      s_cursor[2] = ui;
      s_cursor[3] = i0;
      return ch;
    };
    const int g_cur = s_range[0], g_end = s_range[1];
    if (tid == 0) {
      s_cursor[0] = g_cur;
      s_cursor[1] = g_end;
      s_cursor[2] = g_cur / a.I;
      s_cursor[3] = g_cur - (g_cur / a.I) * a.I;
    }
    if (tid == 0) {
      // count the chunks (same cuts as next_chunk), then describe the first ring's worth
      int nc = 0;
      for (int cur = g_cur, i0 = s_cursor[3]; cur < g_end; ++nc) {
        int nn = g_end - cur;
        if (nn > a.I - i0) nn = a.I - i0;
        const int cap = nc == 0 ? cap0 : P.gu_cap;
        if (nn > cap) nn = cap;
        cur += nn;
        i0 = (i0 + nn == a.I) ? 0 : i0 + nn;
      }
      for (int q = 0; q < kGuSlots && q < nc; ++q) s_chunks[q] = next_chunk(q == 0 ? cap0 : P.gu_cap);
      *reinterpret_cast<int*>(smem + P.chunks + kGuSlots * 12) = nc;
      // the first chunk goes out at once (thread 0 is its only issuer)
      static_assert(kGuFirst == 1, "thread 0 issues the first chunk");
      if (nc > 0) issue_gu_chunk(a, W, T, gu, smem_u32(bars), s_chunks[0]);
    } else if (one && warp == 1) {
      softmax_one(a, T);  // meanwhile
    }
    __syncthreads();
    const int n_chunks = *reinterpret_cast<const int*>(smem + P.chunks + kGuSlots * 12);
    const int n_first = min(kGuFirst, n_chunks), n_ring = min(kGuSlots, n_chunks);
    gu_pend |= (1u << n_first) - 1u;
    // the down prefetch goes out once the first gate/up chunk has landed, so it does not
    // delay that chunk (it is needed only after B2)
    const int iss = mma ? 0 : NT - 32;  // first thread of the issuing warp
    auto issue_dn_prefetch = [&]() {
      if (no > 0) {
        const int nq = min(U, kDnSlots);
        dn_pend |= (1u << nq) - 1u;
        if (tid == iss) {
#pragma unroll 1
          for (int q = 0; q < nq; ++q)
            issue_dn_chunk(a, W, T, dn + q * P.dn_slot, smem_u32(bars + bar_dn0 + q), q, o0, no, codes_room);
        }
      }
    };
    // ---- gate/up ----
    auto gu_loop = [&](auto&& compute) -> bool {
      for (int n = 0; n < n_chunks; ++n) {
        const int q = n % kGuSlots;
        if (!wait_all(q, gu_ph, gu_pend, q)) return false;
        if (n == 0) {
          stamp(a, l, 4);
          gu_pend |= ((1u << n_ring) - 1u) & ~((1u << n_first) - 1u);
          const int qi = tid - iss;
          if (qi >= n_first && qi < n_ring)
            issue_gu_chunk(a, W, T, gu + qi * P.gu_slot, smem_u32(bars + qi), s_chunks[qi]);
          issue_dn_prefetch();
        }
        stamp(a, l, 5);  // (the last chunk's stamp stays)
        const GuChunk c = s_chunks[q];
        const uint8_t* slot = gu + q * P.gu_slot;
        compute(slot, c);
        __syncthreads();  // slot q free again
        if (n + kGuSlots < n_chunks) {
          gu_pend |= 1u << q;
          if (tid == 0) {
            s_chunks[q] = next_chunk(P.gu_cap);
            issue_gu_chunk(a, W, T, gu + q * P.gu_slot, smem_u32(bars + q), s_chunks[q]);
          }
        }
      }
      return true;
    };
    bool gu_ok;
    if (!mma && x_staged && a.R == 1) {
      // one row: the lane's first block of activation pairs lives in registers
      const int NB = a.H >> 5, lane = tid & 31;
      f2_t xr[16];
      if (lane < NB) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const ulonglong2 f = *reinterpret_cast<const ulonglong2*>(s_xp + (size_t)c * NB + lane);
          xr[2 * c] = f.x;
          xr[2 * c + 1] = f.y;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) xr[c] = 0ull;
      }
      gu_ok = gu_loop([&](const uint8_t* slot, const GuChunk& c) {
        gateup_chunk_r1<NBL>(a, T, slot, c, xr, s_xp, s_xs);
      });
    } else {
      gu_ok = gu_loop([&](const uint8_t* slot, const GuChunk& c) {
        if (mma)
          gateup_chunk_mma(a, T, slot, c, x, s_mpart);
        else if (x_staged)
          gateup_chunk<NBL, true>(a, T, slot, c, x, s_xp, s_xs);
        else
          gateup_chunk<NBL, false>(a, T, slot, c, x, s_xp, s_xs);
      });
    }
    if (!gu_ok) return;
    if (n_chunks == 0) {
      stamp(a, l, 4);
      stamp(a, l, 5);
      issue_dn_prefetch();
    }
    // the next layer's router rows can move in now (the GU ring is idle until then)
    if (l + 1 < a.L && router_rows_of_cta(a.E) > 0) {
      router_pend = true;
      if (tid == 0) issue_router_rows(a, a.layer[l + 1].router, s_rw, bar_router);
    }
    stamp(a, l, 6);
    if (!grid_sync(a, sy)) {  // B2: every h written
      bail();
      return;
    }
    stamp(a, l, 7);
    if (mma && no > 0) {
      // ---- wide down: groups of up to 16 of one expert's positions on the tensor cores ----
      const int gpe = (a.R + 15) >> 4;  // position groups per expert
      const int per_e = gpe * kKPartsDn, n_asg = U * per_e;
      stamp(a, l, 8);
      int waited = 0, rel = 0;
      for (int j0 = 0; j0 < n_asg; j0 += NW) {
        const int j1 = min(j0 + NW, n_asg);
        // the round's experts must have landed: one waiting thread per slot
        const int need = (j1 - 1) / per_e + 1;
        if (need > waited) {
          bool ok = true;
          if (tid < need - waited) {
            const int qd = (waited + tid) % kDnSlots;
            ok = mbar_wait_bounded(smem_u32(bars + bar_dn0 + qd), (dn_ph >> qd) & 1u, a.status, a.wait_cycles);
          }
          if (__syncthreads_or(!ok)) {
            bail();
            return;
          }
          for (int u = waited; u < need; ++u) {
            const int qd = u % kDnSlots;
            dn_ph ^= 1u << qd;
            dn_pend &= ~(1u << qd);
          }
          waited = need;
        }
        stamp(a, l, 9);  // (the last round's stamp stays)
        down_round_mma(a, T, dn, P.dn_slot, codes_room, o0, no, j0, n_asg, gpe, s_mpart, s_yall);
        // experts whose groups are all done hand their slots to later experts
        const int rel_new = (j1 < n_asg) ? j1 / per_e : U;
        if (tid < rel_new - rel && rel + tid + kDnSlots < U) {
          const int e = rel + tid, qd = e % kDnSlots;
          issue_dn_chunk(a, W, T, dn + (size_t)qd * P.dn_slot, smem_u32(bars + bar_dn0 + qd), e + kDnSlots, o0, no,
                         codes_room);
        }
        for (int e = rel; e < rel_new; ++e)
          if (e + kDnSlots < U) dn_pend |= 1u << (e % kDnSlots);
        rel = rel_new;
      }
      if (n_asg == 0) stamp(a, l, 9);
      stamp(a, l, 10);
      // each row's picks in rank order
      float* out = a.out + (size_t)l * RH;
      for (int i = tid; i < a.R * no; i += NT) {
        const int r = i / no, ol = i - r * no;
        float acc = 0.f;
        for (int j = 0; j < a.k; ++j) {
          const int pp = T.pick_pos[r * a.k + j];
          if (pp >= 0) acc = __fadd_rn(acc, s_yall[pp * 16 + ol]);
        }
        out[(size_t)r * a.H + o0 + ol] = acc;
      }
    } else if (no > 0) {
      // ---- down: waves of WV consecutive CSR positions, one warp per position ----
      for (int i = tid; i < a.R * kAccStride; i += NT) s_acc[i] = 0.f;
      __syncthreads();
      const int total = T.csr_off[U];
      for (int q = 0; q < 2 && q * WV < total; ++q) {
        h_pend |= 1u << q;
        if (tid == 0) issue_hbatch(a, hslot(q), smem_u32(bars + bar_h0 + q), q * WV, min((q + 1) * WV, total));
      }
      int waited = 0;  // the DN slots of union experts [0, waited) have landed
      int rel = 0;     // union experts [0, rel) are finished and their slots reused
      for (int n = 0, pa = 0; pa < total; ++n, pa += WV) {
        const int pb = min(pa + WV, total);
        const int qh = n & 1;
        if (!wait_all(bar_h0 + qh, h_ph, h_pend, qh)) return;
        if (n == 0) stamp(a, l, 8);
        // the experts of this wave's positions must have landed: one waiting thread per slot
        const int need = T.pos_ui[pb - 1] + 1;
        if (need > waited) {
          bool ok = true;
          if (tid < need - waited) {
            const int qd = (waited + tid) % kDnSlots;
            ok = mbar_wait_bounded(smem_u32(bars + bar_dn0 + qd), (dn_ph >> qd) & 1u, a.status, a.wait_cycles);
          }
          if (__syncthreads_or(!ok)) {
            bail();
            return;
          }
          for (int u = waited; u < need; ++u) {
            const int qd = u % kDnSlots;
            dn_ph ^= 1u << qd;
            dn_pend &= ~(1u << qd);
          }
          waited = need;
        }
        stamp(a, l, 9);  // (the last wave's stamp stays)
        {
          // positions of the wave over the warps; spare warps split a position's rows
          const int npos = pb - pa, wpp = NW / npos;
          const int pi = warp / wpp, part = warp - pi * wpp;
          if (pi < npos) {
            const int pp = pa + pi;
            const int ui = T.pos_ui[pp];
            down_position(a, dn + (size_t)(ui % kDnSlots) * P.dn_slot, codes_room, o0, (part * no) / wpp,
                          ((part + 1) * no) / wpp,
                          reinterpret_cast<const float4*>(hslot(qh) + (size_t)pi * a.I * 4),
                          s_y + pi * kAccStride);
          }
        }
        __syncthreads();
        // combine in CSR order: for each row its experts ascending
        for (int i = tid; i < a.R * no; i += NT) {
          const int r = i / no, ol = i - r * no;
          float acc = s_acc[r * kAccStride + ol];
#pragma unroll 4
          for (int pp = pa; pp < pb; ++pp)
            if (T.pos_row[pp] == r) acc = __fadd_rn(acc, s_y[(pp - pa) * kAccStride + ol]);
          s_acc[r * kAccStride + ol] = acc;
        }
        // experts finished by this wave hand their slots to later experts (one issuing
        // thread per slot)
        const int rel_new = (pb < total) ? T.pos_ui[pb] : U;
        if (tid < rel_new - rel && rel + tid + kDnSlots < U) {
          const int e = rel + tid, qd = e % kDnSlots;
          issue_dn_chunk(a, W, T, dn + (size_t)qd * P.dn_slot, smem_u32(bars + bar_dn0 + qd), e + kDnSlots, o0, no,
                         codes_room);
        }
        for (int e = rel; e < rel_new; ++e)
          if (e + kDnSlots < U) dn_pend |= 1u << (e % kDnSlots);
        rel = rel_new;
        // the wave after next into this h slot
        const int na = pa + 2 * WV;
        if (na < total) {
          h_pend |= 1u << qh;
          if (tid == 0) issue_hbatch(a, hslot(qh), smem_u32(bars + bar_h0 + qh), na, min(na + WV, total));
        }
      }
      __syncthreads();
      stamp(a, l, 10);
      float* out = a.out + (size_t)l * RH;
      for (int i = tid; i < a.R * no; i += NT) {
        const int r = i / no, ol = i - (i / no) * no;
        out[(size_t)r * a.H + o0 + ol] = s_acc[r * kAccStride + ol];
      }
    } else {
      stamp(a, l, 8);
      stamp(a, l, 9);
      stamp(a, l, 10);
    }
    stamp(a, l, 11);
    if (l + 1 < a.L && !grid_sync(a, sy)) {  // B3: layer output complete
      bail();
      return;
    }
    stamp(a, l, 12);  // (the last layer has no B3: its interval is zero)
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
  int32_t tail_rank = 0;
  const void *x = nullptr, *out = nullptr, *stats = nullptr, *ws = nullptr, *stream = nullptr;
  size_t ws_bytes = 0;
  bool operator==(const GraphKey& o) const {
    if (rows != o.rows || tail_rank != o.tail_rank || x != o.x || out != o.out || stats != o.stats ||
        ws != o.ws ||
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
  int32_t tail_rank = 0;
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
  if (w->slot_of_expert && (w->n_slots < 1 || (reinterpret_cast<uintptr_t>(w->slot_of_expert) & 3u)))
    return MOE_EINVAL;
  return MOE_OK;
}

// The dynamic shared-memory limit is an attribute of the kernel function, shared by
// every handle: raise it once to the device's opt-in maximum (minus the kernel's static
// shared memory), so a handle created later with a smaller plan cannot lower it below
// what an earlier handle launches with.
template <int NBL, bool WIDE>
cudaError_t allow_max_dynamic_smem(int device) {
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  cudaFuncAttributes fa{};
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, k_round<NBL, WIDE>);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_round<NBL, WIDE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - (int)fa.sharedSizeBytes);
  return e;
}

// Both kernels of one NBL may serve a handle: raise their limits and check that one CTA
// of each fits an SM with `smem` bytes.
template <int NBL>
cudaError_t prepare_kernels(int device, size_t smem, int& occ) {
  int o1 = 0, o2 = 0;
  cudaError_t e = allow_max_dynamic_smem<NBL, false>(device);
  if (e == cudaSuccess) e = allow_max_dynamic_smem<NBL, true>(device);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o1, k_round<NBL, false>, NT, smem);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o2, k_round<NBL, true>, NT, smem);
  occ = o1 < o2 ? o1 : o2;
  return e;
}

// Rounds of at least kMmaRows rows whose positions and this grid's output rows per CTA fit
// the tensor-core path's shared-memory scratch run on the tensor cores.
bool wide_round(const moe_dims& d, int rows, int grid) {
  const SmemPlan p = smem_plan(d.hidden, d.inter, d.n_experts, d.max_rows, d.top_k, grid);
  return rows >= kMmaRows && rows * d.top_k <= kMmaMaxPos && p.max_orows <= 16;
}

cudaError_t launch_kernel(const cudaLaunchConfig_t& cfg, const RoundArgs& a, bool wide) {
  if (nbl_of(a.H) == 1)
    return wide ? cudaLaunchKernelEx(&cfg, k_round<1, true>, a) : cudaLaunchKernelEx(&cfg, k_round<1, false>, a);
  return wide ? cudaLaunchKernelEx(&cfg, k_round<2, true>, a) : cudaLaunchKernelEx(&cfg, k_round<2, false>, a);
}

size_t smem_bytes(const moe_dims& d, int rows, int grid) {
  return smem_plan(d.hidden, d.inter, d.n_experts, rows, d.top_k, grid).total;
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
  a.Rmax = d.max_rows;
  a.bar = reinterpret_cast<unsigned*>(base + L.ctrl);
  a.logits = reinterpret_cast<float*>(base + L.logits);
  a.hbuf = reinterpret_cast<float*>(base + L.hbuf);
  a.status = h->status;
  a.tail_rank = h->tail_rank;
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
  cfg.dynamicSmemBytes = smem_bytes(h->dims, h->dims.max_rows, h->sm_count);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = launch_kernel(cfg, a, !a.route_only && wide_round(h->dims, a.R, h->sm_count));
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
    a.layer[l].slot = layers[l].slot_of_expert;
    a.layer[l].n_slots = layers[l].n_slots;
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
  const SmemPlan plan = smem_plan(dims->hidden, dims->inter, dims->n_experts, dims->max_rows,
                                  dims->top_k, sms);
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
  e = (nbl_of(dims->hidden) == 1) ? prepare_kernels<1>(device, smem, occ) : prepare_kernels<2>(device, smem, occ);
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

int moe_set_tail_skip(moe_handle* h, int32_t rank) {
  if (!h || rank < 0) return MOE_EINVAL;
  h->tail_rank = rank;
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

int moe_prefill_layer(moe_handle* h, const moe_layer_w* w, const uint16_t* x_bf16, int32_t tokens,
                      float* out, int32_t* expert_counts, void* ws, size_t ws_bytes, void* stream) {
  if (!h) return MOE_EINVAL;
  if (tokens < 1 || tokens > kMaxPrefillTokens || !aligned16(x_bf16) || !aligned16(out) || !aligned16(ws))
    return MOE_EINVAL;
  int rc = check_layer(w);
  if (rc != MOE_OK) return rc;
  if (expert_counts && (reinterpret_cast<uintptr_t>(expert_counts) & 3u)) return MOE_EINVAL;
  const PrefillWs L = prefill_ws_layout(h->dims, tokens);
  if (ws_bytes < L.total) return MOE_EWORKSPACE;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  char* base = static_cast<char*>(ws);
  PrefillArgs a{};
  a.H = h->dims.hidden;
  a.E = h->dims.n_experts;
  a.k = h->dims.top_k;
  a.I = h->dims.inter;
  a.T = tokens;
  a.x = x_bf16;
  a.out = out;
  a.router = w->router;
  a.gu_nib = w->gateup_nib;
  a.gu_sc = w->gateup_scale;
  a.dn_nib = w->down_nib;
  a.dn_sc = w->down_scale;
  a.slot = w->slot_of_expert;
  a.n_slots = w->n_slots;
  a.logits = reinterpret_cast<float*>(base + L.logits);
  a.ids = reinterpret_cast<int*>(base + L.ids);
  a.w = reinterpret_cast<float*>(base + L.w);
  a.counts = reinterpret_cast<int*>(base + L.counts);
  a.offs = reinterpret_cast<int*>(base + L.offs);
  a.cursor = reinterpret_cast<int*>(base + L.cursor);
  a.tiles_gu = reinterpret_cast<int*>(base + L.tiles_gu);
  a.tiles_dn = reinterpret_cast<int*>(base + L.tiles_dn);
  a.pos_tok = reinterpret_cast<int*>(base + L.pos_tok);
  a.pos_pick = reinterpret_cast<int*>(base + L.pos_pick);
  a.pick_pos = reinterpret_cast<int*>(base + L.pick_pos);
  a.hbuf = reinterpret_cast<uint16_t*>(base + L.hbuf);
  a.ybuf = reinterpret_cast<float*>(base + L.ybuf);
  a.user_counts = expert_counts;
  a.status = h->status;
  int launches = 0;
  const int e = prefill_launch(a, &launches, stream);
  h->last_launches = launches;
  return e == (int)cudaSuccess ? MOE_OK : MOE_ECUDA;
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
  key.tail_rank = h->tail_rank;
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
  if (v & kStatusTimeout) return MOE_ETIMEOUT;
  return (v & kStatusBadSlot) ? MOE_EINVAL : MOE_OK;
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
// workspace (grid-barrier words, router logits, exchanged SwiGLU outputs) lives in the file-
// scope array below, which the CUDA runtime places on every device that loads this
// library and keeps until the process exits.  The caller passes only inputs and
// outputs; this path calls no cudaMalloc, cudaFree or allocating library routine.

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;  // 4 MiB per device
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
  (void)smem;  // (checked against the device limit by the caller)
  cudaError_t e = allow_max_dynamic_smem<1, false>(dev);
  if (e == cudaSuccess) e = allow_max_dynamic_smem<1, true>(dev);
  if (e == cudaSuccess) e = allow_max_dynamic_smem<2, false>(dev);
  if (e == cudaSuccess) e = allow_max_dynamic_smem<2, true>(dev);
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
  const size_t smem = smem_bytes(*dims, dims->max_rows, sms);
  const SmemPlan plan =
      smem_plan(dims->hidden, dims->inter, dims->n_experts, dims->max_rows, dims->top_k, sms);
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
  a.Rmax = dd.max_rows;
  a.L = 1;
  a.bar = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + L.ctrl);
  a.logits = reinterpret_cast<float*>(static_cast<char*>(ws) + L.logits);
  a.hbuf = reinterpret_cast<float*>(static_cast<char*>(ws) + L.hbuf);
  a.status = dev_status ? dev_status : own_status;
  a.wait_cycles = kDefaultWaitCycles;
  a.x = x_bf16;
  a.out = out;
  copy_layers(a, w, 1);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the barrier words must start at zero; logits and h are fully overwritten
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
  const cudaError_t e = launch_kernel(cfg, a, wide_round(dd, rows, sms));
  return e == cudaSuccess ? MOE_OK : MOE_ECUDA;
}
